// Internal host-side interface between the C-ABI entry points (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <utility>

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "lily_device.cuh"

namespace lily {

enum GemmMode : int { kModeRouter = 0, kModeGateUp = 1, kModeDown = 2 };

// Arguments of the persistent tcgen05 grouped GEMM (one launch per mode).
//   kModeRouter : logits[t][e] = x[t] . Wr[e] + router_bias[e]      (A = Wr bf16 via TMA)
//   kModeGateUp : h[p][i] = f16(silu(Wg_e x_t)_i * (Wu_e x_t)_i)    (A = dequant(int4), B = fp16 x gathered)
//   kModeDown   : out[t][j] += w * (Wd_e h_p)_j                      (A = dequant(int4), B = h rows)
// Work units are blocks of token rows (the routing block map for routed
// experts, then ceil(T/block_rows) identity blocks for the shared expert) times
// m_tiles pairs of 128-row weight tiles.
struct GemmArgs {
    int mode;
    int T, d, E, top_k, I;
    int bm;               // token rows per block (UMMA N <= 128)
    int K;                // reduction length: d (router, gate/up) or I (down)
    int m_tiles;          // weight-tile pairs per block: 1 (router), I/128 (gate/up), d/256 (down)
    int KT;               // k-steps of 64 per unit, K / 64 rounded up to a multiple of 4
    int n_shared_blocks;  // identity blocks: ceil(T/bm)
    int n_routed_max;     // capacity of block_map
    const int *n_blocks;  // device: routed blocks
    const int *block_map; // device [n][3]: expert, first sorted row, rows
    const int *perm;      // device [T*top_k]
    const float *topk_w;  // device [T*top_k]
    // bf16 scale / bias of the routed (s0,b0: first tile of the pair; s1,b1: second)
    // and shared (ss*, sb*) weights; rows of K/64 groups.
    const uint16_t *s0, *b0, *s1, *b1, *ss0, *sb0, *ss1, *sb1;
    const float *router_bias;
    const __half *xs;        // gate/up B: fp16 x in routing order [(top_k+1)*T][d] (routed rows, then shared)
    float *logits;           // router output [T][E]
    __half *h;               // gate/up output, down input, fp16 [(top_k+1)*T][I]
    float *out;              // down output [T][d], accumulated
    Ctrl *ctrl;
};

// Launches `kernel` as a programmatic dependent of the previous kernel in the
// stream: it may start while that one finishes; it calls pdl_wait before its
// first global memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  Function attributes belong to a device, so this runs once per
// (kernel, device, size); safe to call from several host threads.
cudaError_t set_max_dynamic_smem(const void *kernel, int bytes);

// Dynamic shared memory bytes of grouped_gemm_kernel.
size_t grouped_gemm_smem_bytes();

// Before the expert GEMMs: xs = fp16(x) in routing order (routed rows by perm,
// then the T shared-expert rows), [(top_k+1)*T][d], written token by token from
// inv = the inverse of perm.  (out is zeroed by the gate/up GEMM launch.)
cudaError_t launch_prep_experts(const uint16_t *x, const int *inv, __half *xs, int T, int d, int top_k, int *status,
                                cudaStream_t stream);
// inv[perm[p]] = p for p < T*top_k (when the routing tables come from elsewhere).
cudaError_t launch_invert_perm(const int *perm, int *inv, int n, int *status, cudaStream_t stream);

// tmB: B operand rows (x for the router, xs for gate/up, h for down).
// tmA0/tmA1: routed weight maps of the two 128-row tiles (router: Wr for both);
// tmSA0/tmSA1: shared-expert weight maps.
cudaError_t launch_grouped_gemm(const GemmArgs &g, const CUtensorMap &tmB, const CUtensorMap &tmA0,
                                const CUtensorMap &tmA1, const CUtensorMap &tmSA0, const CUtensorMap &tmSA1,
                                int grid, cudaStream_t stream);

// Routing: top-k + per-chunk histogram (+ last-block scan and block map), then scatter.
struct RouteArgs {
    int T, E, top_k, bm;
    const float *logits;
    int *topk_idx;
    float *topk_w;
    int *counts, *offsets, *perm, *block_map, *n_blocks;
    int *inv;           // [T*top_k]: row of assignment t*top_k + j (inverse of perm), or NULL
    int *chunk_counts;  // [C][E]
    int *chunk_base;    // [C][E]: chunk's first row within its expert (relative to offsets[e])
    int n_chunks;
    Ctrl *ctrl;
};
constexpr int kRouteChunkTokens = 32;
cudaError_t launch_topk_count(const RouteArgs &a, cudaStream_t stream);
cudaError_t launch_route_scan(const RouteArgs &a, cudaStream_t stream);
cudaError_t launch_scatter(const RouteArgs &a, cudaStream_t stream);

// Decode path (1 <= T <= 8): one persistent cooperative kernel runs a chain of
// layers; the layers hand their data to each other through tagged words in the
// workspace (see decode.cu).
struct DecodeLayerPtrs {
    const uint16_t *router_w;
    const float *router_bias;
    const uint8_t *gate_q, *up_q, *down_q;
    const uint16_t *gate_s, *gate_b, *up_s, *up_b, *down_s, *down_b;
    const uint8_t *sh_gate_q, *sh_up_q, *sh_down_q;
    const uint16_t *sh_gate_s, *sh_gate_b, *sh_up_s, *sh_up_b, *sh_down_s, *sh_down_b;
};
constexpr int kDecodeLayersPerLaunch = 20;  // layer table passed as a kernel parameter (<= 4 KB)
constexpr int kDecodeMaxT = 8;
constexpr int kDecodeMaxUnits = 8 * kDecodeMaxT + 1;  // distinct routed experts of 8 tokens + the shared one
// Ready counters of one layer: [0] CTAs whose router rows are written, [1] down
// tasks whose output rows are written, [2 + u] gate/up tasks of unit u written.
constexpr int kDecodeReadySlots = 2 + kDecodeMaxUnits;

struct DecodeArgs {
    int T, d, E, top_k, I;
    int layer0, n_layers;   // this launch runs global layers [layer0, layer0 + n_layers)
    int last_launch;        // the call's last launch: also exports x_next of its last layer
    int n_slots, slot_bytes;
    const uint16_t *x_in;   // bf16 [T][d]: input of global layer 0
    float *out;             // f32 [total layers][T][d]
    uint16_t *x_next;       // bf16 [total layers][T][d] or NULL
    float *trace_logits;    // [total layers][T][E] or NULL
    int *trace_idx;         // [total layers][T][top_k] or NULL
    float *trace_w;         // [total layers][T][top_k] or NULL
    // exchange area in the workspace: data double buffered by layer parity,
    // per-layer ready counters (zeroed before the first launch of a call)
    float *logits_x;        // [2][T][E] router logits
    uint32_t *h_x;          // [2][kDecodeMaxUnits][I/128][T][4][16] h' pairs in the down projection's B layout
    float *out_x;           // [2][T][d] layer outputs
    unsigned int *ready;    // [layers of the call][kDecodeReadySlots]
    int *abort_flag;        // raised by the CTA whose wait ran out; the others give up too
    Ctrl *ctrl;
    DecodeLayerPtrs L[kDecodeLayersPerLaunch];
};
static_assert(sizeof(DecodeArgs) <= 4096, "decode kernel parameters stay within 4 KB");
// Ring slots that fit next to the fixed shared memory for this shape (0: the
// shape does not fit), the bytes of one slot, and the dynamic shared memory of
// the launch.
int decode_ring_slots(int T, int d, int I);
int decode_launch_slots(int T, int d, int I);  // device-checked (needs the device current)
int decode_slot_bytes(int d, int I);
size_t decode_smem_bytes(int T, int d, int I, int n_slots);
cudaError_t launch_decode(const DecodeArgs &a, int grid, cudaStream_t stream);

}  // namespace lily
