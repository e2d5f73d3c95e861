/*
 * lily_moe.h -- C ABI of the GB300 (sm_103a) mixture-of-experts layer library
 * (liblily_moe.so).
 *
 * The layer is the one described on the page "Perplexity libera o Lily"
 * (noticiai.com.br):
 *   - section "O modelo em tres formatos de carga": a router scores 256 experts
 *     and selects eight, plus one shared expert that sees every token; the
 *     experts form uneven groups of tokens;
 *   - section "Prefill e decode: onde estao os ganhos": weights are 4-bit
 *     group-wise affine (each group of 64 weights shares one bf16 scale and one
 *     bf16 bias), rebuilt to bf16 one tile at a time inside the grouped GEMM
 *     with FP32 accumulation; the routing histogram, prefix scan, scatter and
 *     block map stay on the GPU with no CPU synchronisation inside the layer;
 *     at batch 1 (decode) bandwidth sets the ceiling.
 *
 * Conventions shared by every entry point
 *   - Every pointer marked "device" is CUDA device memory owned by the caller.
 *     The library allocates nothing and frees nothing on these calls.
 *   - Every call is asynchronous on `stream`: it validates its arguments on the
 *     host, enqueues kernels and returns.  No call synchronises or copies data
 *     to the host, except lily_moe_device_status().  Because a call enqueues
 *     only stream work, it may be recorded into the caller's CUDA graph by
 *     stream capture (see lily_moe_route_noalloc for its one exception).
 *   - Every device pointer must be 16-byte aligned.
 *   - Return value: LILY_OK (0) or a negative LILY_ERR_* code.  Host-side errors
 *     are returned before anything is enqueued.  Errors detected by a kernel
 *     (a device wait that timed out, an index out of range, a value beyond the
 *     fp16 range) are written, first one wins, into a status word at the start
 *     of the workspace and are read with lily_moe_device_status().
 *   - T = 0 is valid and enqueues nothing.
 *   - Inputs are assumed finite; NaN or Inf inputs give unspecified results.
 *   - Range: the expert GEMMs run on fp16 operands (the rebuilt weights, x and
 *     the SwiGLU product h; fp32 accumulation).  Every |x| and every |h| =
 *     |silu(gate x) * (up x)| must stay below 65520, which rounds to the fp16
 *     maximum 65504; a larger finite value would become infinite.  The kernels
 *     check every converted x and h value and record LILY_ERR_DEVICE_RANGE in
 *     the status word when one overflows (the outputs of that call are then
 *     unspecified).  The router logits are computed from bf16 x in fp32 and
 *     have no such limit.
 *   - lily_moe_forward / lily_moe_grouped_gemm: the routing tables and logits
 *     are bit-reproducible from run to run; the layer output is not: the down
 *     projection adds each token's nine weighted expert rows into `out` with
 *     fp32 atomic adds whose order varies, so `out` may differ between runs in
 *     its last bits.  lily_moe_decode is bit-reproducible.
 *   - bf16 values are passed as their uint16 bit patterns.
 *   - A workspace must not be shared by calls that may run concurrently.
 */
#ifndef LILY_MOE_H
#define LILY_MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    LILY_OK = 0,
    LILY_ERR_INVALID = -1,        /* null pointer, negative size, inconsistent arguments */
    LILY_ERR_UNSUPPORTED = -2,    /* shape outside the supported set (see lily_moe_shape) */
    LILY_ERR_MISALIGNED = -3,     /* a device pointer is not 16-byte aligned */
    LILY_ERR_WORKSPACE = -4,      /* workspace smaller than lily_moe_workspace_bytes() */
    LILY_ERR_LAUNCH = -5,         /* a CUDA call failed while enqueueing */
    LILY_ERR_DEVICE_TIMEOUT = -6, /* a kernel's bounded wait ran out (device-detected) */
    LILY_ERR_DEVICE_INDEX = -7,   /* a kernel saw an index out of range (device-detected) */
    LILY_ERR_SCRATCH_LIMIT = -8,  /* size above the fixed scratch of lily_moe_route_noalloc */
    LILY_ERR_DEVICE_RANGE = -9    /* a value beyond the fp16 range of the expert GEMMs (device-detected) */
};

/*
 * Layer shape.  Supported set:
 *   E = 256, top_k = 8, group = 64,
 *   d a multiple of 256 in [256, 16384], I a multiple of 128 in [128, 4096],
 *   I_shared = I, block_rows in {16, 32, 64, 128}, 0 <= T <= 1048576.
 * lily_moe_decode additionally needs 1 <= T <= 8, d <= 4096 and I <= 1024.
 */
typedef struct lily_moe_shape {
    int32_t T;          /* tokens */
    int32_t d;          /* hidden size */
    int32_t E;          /* routed experts */
    int32_t top_k;      /* experts selected per token */
    int32_t I;          /* routed-expert intermediate size */
    int32_t I_shared;   /* shared-expert intermediate size */
    int32_t group;      /* quantisation group along the reduction dimension */
    int32_t block_rows; /* rows per block-map entry (tile height of the grouped GEMM) */
} lily_moe_shape;

/*
 * One 4-bit group-affine matrix W [rows][K] (device, read-only):
 *   q     uint8 [rows][K/2]; element k of row n is in byte q[n][k/2],
 *         LOW nibble for even k, HIGH nibble for odd k (unsigned 0..15);
 *   scale bf16  [rows][K/64];  bias bf16 [rows][K/64];
 *   W[n][k] = q[n][k] * scale[n][k/64] + bias[n][k/64].
 */
typedef struct lily_q4 {
    const uint8_t *q;
    const uint16_t *scale;
    const uint16_t *bias;
} lily_q4;

/*
 * One layer's weights (device, read-only).
 *   router_w     bf16 [E][d]
 *   router_bias  f32 [E], or NULL; added to the logits before selection and softmax
 *   gate, up     routed experts stacked by expert: rows E*I, K = d
 *                (expert e owns rows [e*I, (e+1)*I))
 *   down         routed experts stacked by expert: rows E*d, K = I
 *   sh_gate, sh_up  shared expert: rows I_shared, K = d
 *   sh_down         shared expert: rows d, K = I_shared
 * Each expert is SwiGLU: y = down( silu(gate x) * (up x) ), silu(z) = z / (1 + e^-z).
 */
typedef struct lily_moe_weights {
    const uint16_t *router_w;
    const float *router_bias;
    lily_q4 gate, up, down;
    lily_q4 sh_gate, sh_up, sh_down;
} lily_moe_weights;

/*
 * Routing tables (device, caller-owned, written by lily_moe_route; read by
 * lily_moe_grouped_gemm).  Sizes for T tokens:
 *   logits    f32 [T][E], or NULL (then kept in the workspace)
 *   topk_idx  int32 [T][top_k]  selected experts, by descending logit, lower
 *                               index first among equal logits
 *   topk_w    f32 [T][top_k]    softmax over E renormalised over the top_k
 *                               (= softmax over the selected logits)
 *   counts    int32 [E]         tokens per expert (histogram)
 *   offsets   int32 [E+1]       exclusive scan of counts; offsets[E] = T*top_k
 *   perm      int32 [T*top_k]   expert-sorted order: perm[offsets[e] + r] =
 *                               t*top_k + j for the r-th assignment of expert e
 *                               in ascending token order (stable scatter)
 *   block_map int32 [capacity][3] (expert, first sorted row, rows) for each
 *                               block of at most block_rows rows, experts
 *                               ascending; capacity from lily_moe_block_capacity()
 *   n_blocks  int32 [1]         number of valid block_map entries
 */
typedef struct lily_moe_routing {
    float *logits;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *counts;
    int32_t *offsets;
    int32_t *perm;
    int32_t *block_map;
    int32_t *n_blocks;
} lily_moe_routing;

/*
 * Optional per-layer record of the decode path (device, caller-owned); any
 * member may be NULL.  logits f32 [n_layers][T][E]; topk_idx int32
 * [n_layers][T][top_k]; topk_w f32 [n_layers][T][top_k].
 */
typedef struct lily_moe_decode_trace {
    float *logits;
    int32_t *topk_idx;
    float *topk_w;
} lily_moe_decode_trace;

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int lily_moe_version(void);

/* Human-readable text of a LILY_* code (static storage, never NULL). */
const char *lily_moe_status_string(int status);

/*
 * The CUDA error behind the last LILY_ERR_LAUNCH returned on the calling
 * thread: which step failed and the CUDA error name and text ("" if none).
 * Thread-local storage, valid until the thread's next failing call.
 */
const char *lily_moe_last_error_detail(void);

/* Shape check only: LILY_OK or LILY_ERR_INVALID / LILY_ERR_UNSUPPORTED. */
int lily_moe_check_shape(const lily_moe_shape *shape);

/* Entries a routing block_map must hold: min(T*top_k, E + ceil(T*top_k/block_rows)), at least 1. */
int64_t lily_moe_block_capacity(const lily_moe_shape *shape);

/*
 * Workspace bytes needed by the calls below for this shape: the maximum over
 * lily_moe_route / lily_moe_grouped_gemm / lily_moe_forward (T tokens) and, if
 * n_layers_decode > 0, lily_moe_decode.  Returns 0 for an unsupported shape.
 * The workspace is device memory, 256-byte aligned, caller-owned; its first
 * bytes hold the sticky device status word (see lily_moe_clear_status).
 */
size_t lily_moe_workspace_bytes(const lily_moe_shape *shape, int32_t n_layers_decode);

/*
 * Routing (steps: router logits, top-k + weights, histogram, exclusive scan,
 * stable scatter, block map), all on the GPU on `stream`, no host sync.
 * x: bf16 [T][d] device.  r: every member except r->logits must be non-NULL.
 * When the 64-token blocks are fewer than the SMs, the router GEMM also splits
 * the reduction over d (up to 8 parts, chosen from the shape alone) and the
 * top-8 kernel adds the parts in a fixed order, so the logits stay
 * bit-reproducible.
 */
int lily_moe_route(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                   lily_moe_routing *r, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Grouped expert GEMMs from given routing tables: for every expert block, the
 * gate/up GEMM with the 4-bit weights dequantised to fp16 inside the GEMM, SwiGLU,
 * then the down GEMM whose epilogue scales by topk_w and adds into token order;
 * the shared expert is added with weight 1.  out: f32 [T][d] device, overwritten.
 * r: topk_w, perm, block_map and n_blocks are read (must be non-NULL).
 */
int lily_moe_grouped_gemm(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                          const lily_moe_routing *r, float *out, void *ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * The whole layer: lily_moe_route then lily_moe_grouped_gemm.  r may be NULL
 * (routing tables then live in the workspace).
 */
int lily_moe_forward(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                     float *out, lily_moe_routing *r, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * lily_moe_forward with stage timing: if `events` is non-NULL it must hold 6
 * created CUDA events, recorded on `stream` at: start, after the router GEMM,
 * after the routing tables, after the routing-order copy of x, after the
 * gate/up GEMM (which also zeroes out), after the down GEMM.
 */
int lily_moe_forward_timed(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                           float *out, lily_moe_routing *r, void *ws, size_t ws_bytes,
                           cudaStream_t stream, cudaEvent_t *events);

/*
 * Decode: n_layers MoE layers back to back on T (1..8) tokens.
 *   layers     HOST array of n_layers weight structs (device pointers inside)
 *   x          bf16 [T][d] device: input of layer 0
 *   out        f32 [n_layers][T][d] device: out[l] = layer l's output
 *   x_next     bf16 [n_layers][T][d] device or NULL:
 *              x_next[l] = bf16( out[l] / sqrt(mean_c out[l][t][c]^2 + 1e-6) ),
 *              the input of layer l+1 (a parameter-free RMS norm standing in
 *              for the attention / recurrent blocks between MoE layers)
 *   trace      optional per-layer routing record, or NULL
 * The launches (three kernels per layer) are recorded once into a CUDA graph
 * cached by argument values and replayed (unless `stream` is already
 * capturing, then they are enqueued directly).  The result is bit-reproducible
 * from run to run (no atomics; fixed summation order).
 */
int lily_moe_decode(const lily_moe_shape *shape, int32_t n_layers, const lily_moe_weights *layers,
                    const uint16_t *x, float *out, uint16_t *x_next,
                    const lily_moe_decode_trace *trace, void *ws, size_t ws_bytes,
                    cudaStream_t stream);

/*
 * Reads the workspace's sticky device status word: synchronises `stream`,
 * copies 4 bytes to the host.  Returns LILY_OK, a LILY_ERR_DEVICE_* code, or
 * LILY_ERR_LAUNCH if the stream itself reports an error.
 */
int lily_moe_device_status(const void *ws, cudaStream_t stream);

/* Enqueues a reset of the workspace's status word to LILY_OK. */
int lily_moe_clear_status(void *ws, cudaStream_t stream);

/*
 * Grouped-query decode attention over a fixed-block KV cache: one decode step
 * of the model's full-attention layers for B sequences.
 *
 * Method: the page "Perplexity libera o Lily" (noticiai.com.br), section "O
 * modelo em tres formatos de carga" (grouped-query attention, 16 query heads
 * over two KV heads, a growing KV cache) and section "Prefill e decode: onde
 * estao os ganhos" (query heads of a KV head packed together, coalesced cache
 * reads, a fixed-block cache layout).  For each sequence b and query head h,
 * with group = H_q / H_kv and g = h / group:
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_g[t]) V_g[t],
 * over the sequence's tokens t < seq_lens[b]; K_g[t] / V_g[t] is row t % bs of
 * cache block block_table[b][t / bs], KV head g.  Computed with bf16 inputs,
 * fp32 scores and accumulation; the softmax weights are rounded to bf16 before
 * they multiply V (their sum is taken over the rounded values).
 *
 * Layouts (row-major, device memory, all 16-byte aligned):
 *   q         bf16 [B][H_q][D] (positional rotation already applied)
 *   k_cache   bf16 [n_cache_blocks][H_kv][block_size][D]; v_cache the same
 *   block_table int32 [B][max_blocks]: physical block of each logical block
 *   seq_lens  int32 [B]: tokens in each sequence's cache, 0..max_blocks*block_size
 *   out       f32 [B][H_q][D]; a sequence with no tokens gets zeros
 * Supported: D in {64, 128, 256}; block_size in {32, 64, 128} with
 * block_size * D <= 16384; H_q % H_kv == 0 and H_q / H_kv <= 8;
 * n_cache_blocks * H_kv * block_size < 2^31.
 * Device-detected: a used table entry outside [0, n_cache_blocks) or a length
 * outside [0, max_blocks * block_size] records LILY_ERR_DEVICE_INDEX (read it
 * with lily_moe_device_status on the same workspace); the kernels then read
 * block 0 / clamp the length instead.
 * Enqueues two kernels (split and combine) on `stream`; no host sync.  The
 * result is bit-reproducible from run to run.
 */
typedef struct lily_attn_shape {
    int32_t B;           /* sequences */
    int32_t H_q, H_kv;   /* query heads, KV heads */
    int32_t D;           /* head dimension */
    int32_t block_size;  /* tokens per cache block */
    int32_t max_blocks;  /* columns of block_table */
} lily_attn_shape;

/* Workspace bytes of lily_attn_decode (0: unsupported shape). */
size_t lily_attn_workspace_bytes(const lily_attn_shape *shape);

/* scale: multiplies q . k (1 / sqrt(D) for plain scaled dot-product attention). */
int lily_attn_decode(const lily_attn_shape *shape, const uint16_t *q, const uint16_t *k_cache,
                     const uint16_t *v_cache, int64_t n_cache_blocks, const int32_t *block_table,
                     const int32_t *seq_lens, float scale, float *out, void *ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * Gated DeltaNet scan: the fixed-size recurrence of the model's linear-attention
 * layers over T tokens of one sequence, the state kept in registers.
 *
 * Method: the page "Perplexity libera o Lily" (noticiai.com.br), section "O
 * modelo em tres formatos de carga" (30 Gated DeltaNet layers, a recurrence of
 * fixed size) and section "Prefill e decode: onde estao os ganhos" (a scan with
 * its state in registers).  The page gives no formula; this is the gated delta
 * rule.  Per value head h (key head h / (H_v / H_k)), state S (d_v x d_k):
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *   o_t = scale * S_t q_t
 * The normalisation, gating and convolution that produce q, k, v, alpha and
 * beta come before the scan and are the caller's.  fp32 state and arithmetic.
 *
 * Layouts (row-major, device memory, 16-byte aligned):
 *   q, k   bf16 [T][H_k][d_k];  v  bf16 [T][H_v][d_v]
 *   alpha, beta  f32 [T][H_v]
 *   state_in     f32 [H_v][d_v][d_k], or NULL for a zero state
 *   out          f32 [T][H_v][d_v];  state_out  f32 [H_v][d_v][d_k] (may not
 *                alias state_in)
 * Supported: d_k in {64, 128}; d_v a multiple of 16 in [16, 1024];
 * H_v % H_k == 0; T >= 0 (T = 0 copies the state; the token arrays may then
 * be NULL).  One kernel on `stream`; bit-reproducible.
 */
typedef struct lily_gdn_shape {
    int32_t T;          /* tokens */
    int32_t H_k, H_v;   /* query/key heads, value heads */
    int32_t d_k, d_v;   /* key and value head sizes */
} lily_gdn_shape;

int lily_gdn_scan(const lily_gdn_shape *shape, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *alpha, const float *beta, const float *state_in, float scale, float *out,
                  float *state_out, cudaStream_t stream);

/*
 * Routing without a caller workspace.  The method has no counterpart: this entry
 * point exists for callers that may not allocate device memory when they call
 * the layer, e.g. a plugin that runs inside another engine's fixed memory
 * budget, or a serving loop that forbids device allocation after start-up, and
 * so cannot provide the workspace that lily_moe_route needs.
 *
 * It computes exactly what lily_moe_route computes (same kernels, same
 * results), but keeps its scratch (per-chunk expert counts, their scanned
 * write offsets, the last-block counter, the status word and the router's
 * partial logits) in a fixed array that the library holds in device memory on
 * every GPU that loads it, LILY_NOALLOC_SCRATCH_BYTES bytes (about 10.5 MB),
 * for the life of the process.
 *   - T must be <= LILY_NOALLOC_MAX_TOKENS, else LILY_ERR_SCRATCH_LIMIT.
 *   - r->logits must be non-NULL (the logits are an output here, not scratch).
 *   - device_status: device int32 or NULL; if given, the call's device status
 *     (LILY_OK or a LILY_ERR_DEVICE_* code) is copied there on `stream` at the
 *     end (T = 0: LILY_OK is written there).  The scratch status word is
 *     cleared at the start of every call.
 *   - The first call in a CUDA context looks up the array's device address
 *     (no allocation; again after a device reset, which creates a new
 *     context); make that first call outside any stream capture.
 *   - Every call on a device shares the one array: calls that may overlap on
 *     the GPU (other streams, other threads) race and must be serialised by the
 *     caller.
 * Allocates nothing: no cudaMalloc, no cudaFree, no library allocation.
 */
#define LILY_NOALLOC_MAX_TOKENS 8192
/* control block, two per-chunk tables of 256 int32 per 32 tokens, then the
 * router's partial logits when it splits K (at most 152 x 64 token rows of 256
 * fp32 partial logits) */
#define LILY_NOALLOC_SCRATCH_BYTES \
    (256 + 2 * 4 * 256 * (LILY_NOALLOC_MAX_TOKENS / 32) + 256 + 4 * 256 * 152 * 64)
int lily_moe_route_noalloc(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                           lily_moe_routing *r, int32_t *device_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LILY_MOE_H */
