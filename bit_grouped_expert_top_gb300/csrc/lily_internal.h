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
// m_tiles pairs of 128-row weight tiles.  The router may also split K: unit
// (block, split s) takes blocks [s KB / ksplit, (s + 1) KB / ksplit) of the KB
// four-k-step blocks of K and writes its partial logits (no bias) to
// logits_part[s]; the top-8 kernel adds the splits in order and the bias.
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
    float *logits;           // router output [T][E] (ksplit == 1)
    int ksplit;              // router: K splits (1 <= ksplit <= KT / 4); expert modes: 1
    float *logits_part;      // router, ksplit > 1: partial logits [ksplit][T][E]
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

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (never lowers it: the limit is the largest size asked for in
// this context).  Safe to call from several host threads.
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
    // ksplit == 1: the router wrote the logits (bias included).  ksplit > 1: the
    // router wrote ksplit partial sums; the top-8 kernel adds them in split order,
    // then the bias, and writes the logits.
    float *logits;              // [T][E]
    int ksplit;
    const float *logits_part;   // [ksplit][T][E]
    const float *router_bias;   // [E] or NULL
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
// Tokens per routing chunk: 32, fewer for small T (more CTAs in the one-launch
// path), and the number of chunks.
inline int route_chunk_tokens(int64_t T) { return T <= 512 ? 8 : T <= 1024 ? 16 : kRouteChunkTokens; }
inline int64_t route_chunks(int64_t T)
{
    const int ct = route_chunk_tokens(T);
    return T > 0 ? (T + ct - 1) / ct : 1;
}
constexpr int kMaxRouterSplit = 8;  // router K splits (partial logits summed by the top-8 kernel)
cudaError_t launch_topk_count(const RouteArgs &a, cudaStream_t stream);
// All three steps in one launch (n_chunks <= kRouteFusedChunks).
constexpr int kRouteFusedChunks = 64;
cudaError_t launch_route_fused(const RouteArgs &a, cudaStream_t stream);
cudaError_t launch_route_scan(const RouteArgs &a, cudaStream_t stream);
cudaError_t launch_scatter(const RouteArgs &a, cudaStream_t stream);

// Decode path (1 <= T <= 8).
struct DecodeLayerArgs {
    int T, d, E, top_k, I, layer;
    const uint16_t *router_w;
    const float *router_bias;
    const uint8_t *gate_q, *up_q, *down_q;
    const uint16_t *gate_s, *gate_b, *up_s, *up_b, *down_s, *down_b;
    const uint8_t *sh_gate_q, *sh_up_q, *sh_down_q;
    const uint16_t *sh_gate_s, *sh_gate_b, *sh_up_s, *sh_up_b, *sh_down_s, *sh_down_b;
    const uint16_t *x_in;     // layer 0 input bf16 [T][d] (NULL for later layers)
    const float *prev_out;    // previous layer output f32 [T][d] (NULL for layer 0)
    float *out;               // this layer's output f32 [T][d]
    uint16_t *x_export;       // bf16 [T][d] or NULL: normalised input of this layer (x_next of the previous)
    float *trace_logits;      // [T][E] or NULL
    int *trace_idx;           // [T][top_k] or NULL
    float *trace_w;           // [T][top_k] or NULL
    // workspace
    uint16_t *x_cur;          // bf16 [T][d]
    __half *xp;               // fp16 [8][d] layer input in the permuted B layout of the expert GEMVs (tokens >= T zero)
    float *logits;            // [T][E]
    int *n_units;             // [1]: distinct experts used + 1 (shared last)
    int *unit_expert;         // [top_k*T+1]
    int *unit_mask;           // [top_k*T+1] token bitmask
    float *unit_w;            // [top_k*T+1][8]
    __half *h;                // fp16 [top_k*T+1][8][I]
    Ctrl *ctrl;
};
cudaError_t launch_decode_layer(const DecodeLayerArgs &a, int num_sms, cudaStream_t stream);

// Grouped-query decode attention over a fixed-block KV cache (attention.cu).
// Split-K: CTA (split s, KV head g, sequence b) takes the cache blocks
// [s nblk / S, (s + 1) nblk / S) of sequence b and all query heads of group g,
// and writes an unnormalised partial (running max in log2 units, sum of
// weights, weighted sum of values); the combine kernel merges the splits.
struct AttnArgs {
    int B, H_q, H_kv, D, bs, max_blocks, n_splits, group;
    long long n_cache_blocks;
    float scale_log2;           // scale * log2(e)
    const uint16_t *q;          // bf16 [B][H_q][D]
    const int *block_table;     // [B][max_blocks]
    const int *seq_lens;        // [B]
    float *part_ml;             // [B][H_kv][S][8][2]: max (log2 units), sum of weights
    float *part_acc;            // [B][H_kv][S][8][D]
    float *out;                 // [B][H_q][D]
    Ctrl *ctrl;
};
constexpr int kAttnMaxGroup = 8;    // query heads per KV head (the N = 8 side of the MMA)
constexpr int kAttnMaxSplits = 256; // splits per (sequence, KV head)
// Ring stages of K+V block tiles for this shape (0: unsupported), and the
// dynamic shared memory of the split kernel.
int attn_stages(int D, int bs);
size_t attn_smem_bytes(int D, int bs);
// tmK / tmV: the caches as 2-D bf16 [n_blocks * H_kv * bs][D], box 64 x bs, 128-byte swizzle.
cudaError_t launch_attn_decode(const AttnArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t stream);

// Gated DeltaNet scan (gdn.cu): CTA (16-row slice of the state, value head).
struct GdnArgs {
    int T, H_k, H_v, d_k, d_v;
    float scale;
    const uint16_t *q, *k;     // bf16 [T][H_k][d_k]
    const uint16_t *v;         // bf16 [T][H_v][d_v]
    const float *alpha, *beta; // [T][H_v]
    const float *state_in;     // [H_v][d_v][d_k] or NULL (zeros)
    float *out;                // [T][H_v][d_v]
    float *state_out;          // [H_v][d_v][d_k]
};
size_t gdn_smem_bytes(int d_k);
cudaError_t launch_gdn_scan(const GdnArgs &a, cudaStream_t stream);

}  // namespace lily
