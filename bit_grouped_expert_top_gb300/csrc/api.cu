// C-ABI entry points of liblily_moe.so (declared in include/lily_moe.h):
// argument validation, workspace carving, TMA tensor-map encoding and the
// launch sequence of each call.  No entry point allocates device memory or
// synchronises, except lily_moe_device_status.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "lily_internal.h"
#include "lily_moe.h"

namespace {
unsigned long long current_context_id();
}  // namespace

namespace lily {
cudaError_t launch_decode_final_norm(const float *prev_out, uint16_t *x_export, int T, int d, cudaStream_t stream);

cudaError_t set_max_dynamic_smem(const void *kernel, int bytes)
{
    // The attribute only ever grows: a launch with less shared memory than the
    // limit is fine, so the largest size asked for so far is what is set.
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, unsigned long long>, int> set_to;  // (kernel, device, context)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx_id = current_context_id();
    const auto key = std::make_tuple(kernel, dev, ctx_id);
    std::lock_guard<std::mutex> lock(mu);
    auto it = set_to.find(key);
    if (it != set_to.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && ctx_id != 0) set_to[key] = bytes;
    return e;
}
}  // namespace lily

namespace {

using namespace lily;

constexpr int kVersion = 10100;  // 1.1.0

// Unique id of the CUDA context current on this thread (the runtime's primary
// context of the current device), 0 if none is current yet.  Caches of
// per-context state (symbol addresses, kernel attributes, instantiated graphs)
// are keyed by it:
// after cudaDeviceReset the device gets a new context with a new id, so no
// entry made in the old context is used again.
// The two driver calls are looked up through the runtime (the library does
// not link the driver library, so it still loads on a machine without one).
unsigned long long current_context_id()
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrentFn>(p);
            get_id = reinterpret_cast<GetIdFn>(q);
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ workspace layouts
struct PrefillLayout {
    size_t ctrl, chunk_counts, chunk_base, h, xs, inv, logits, idx, w, counts, offsets, perm, block_map, n_blocks, total;
};

int64_t block_capacity(const lily_moe_shape &s)
{
    const int64_t a = static_cast<int64_t>(s.T) * s.top_k;
    return std::max<int64_t>(1, std::min<int64_t>(a, s.E + ceil_div(a, s.block_rows)));
}

// k-steps of 64 of the grouped GEMM for reduction length K: K / 64 rounded up
// to whole blocks of four (the kernel reads zeros past K).
int gemm_k_steps(int64_t K)
{
    return static_cast<int>(((K / 64) + 3) / 4 * 4);
}

// Router K splits: about one unit (64 tokens x a share of K) per SM of a
// 152-SM GPU while the token blocks alone are fewer, at most 8 and at most one
// per block of four k-steps.  A fixed budget (not the device's SM count) keeps
// the logits' rounding a function of the shape alone.
constexpr int kRouterUnitBudget = 152;
constexpr int kRouterBlockRows = 64;

int router_ksplit(const lily_moe_shape &s)
{
    const int64_t blocks = std::max<int64_t>(1, ceil_div(s.T, kRouterBlockRows));
    const int64_t kb = gemm_k_steps(s.d) / 4;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({kMaxRouterSplit, kb, kRouterUnitBudget / blocks})));
}

// Bytes of the router's partial logits (0 without a split).
size_t router_part_bytes(const lily_moe_shape &s)
{
    const int k = router_ksplit(s);
    return k > 1 ? static_cast<size_t>(k) * s.T * s.E * 4 : 0;
}

PrefillLayout prefill_layout(const lily_moe_shape &s)
{
    PrefillLayout L{};
    const int64_t T = s.T, E = s.E, k = s.top_k;
    const int64_t C = route_chunks(T);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + std::max<size_t>(bytes, 1));
        return at;
    };
    L.ctrl = take(sizeof(Ctrl));
    L.chunk_counts = take(C * E * 4);
    L.chunk_base = take(C * E * 4);
    L.h = take((k + 1) * T * s.I * 2);
    // xs also holds the router's partial logits before the prep kernel writes it
    L.xs = take(std::max<size_t>((k + 1) * T * s.d * 2, router_part_bytes(s)));
    L.inv = take(T * k * 4);
    L.logits = take(T * E * 4);
    L.idx = take(T * k * 4);
    L.w = take(T * k * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(T * k * 4);
    L.block_map = take(block_capacity(s) * 3 * 4);
    L.n_blocks = take(4);
    L.total = off;
    return L;
}

struct DecodeLayout {
    size_t ctrl, x_cur, xp, logits, n_units, unit_expert, unit_mask, unit_w, h, total;
};

DecodeLayout decode_layout(const lily_moe_shape &s)
{
    DecodeLayout L{};
    const int64_t T = s.T, U = static_cast<int64_t>(s.top_k) * s.T + 1;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + std::max<size_t>(bytes, 1));
        return at;
    };
    L.ctrl = take(sizeof(Ctrl));
    L.x_cur = take(T * s.d * 2);
    L.xp = take(8 * s.d * 2);  // fp16 layer input, 8 token columns, permuted for the tensor-core GEMV
    L.logits = take(T * s.E * 4);
    L.n_units = take(4);
    L.unit_expert = take(U * 4);
    L.unit_mask = take(U * 4);
    L.unit_w = take(U * 8 * 4);
    L.h = take(U * 8 * s.I * 2);
    L.total = off;
    return L;
}

// ------------------------------------------------------------------ decode attention
int attn_check_shape(const lily_attn_shape *s)
{
    if (!s) return LILY_ERR_INVALID;
    if (s->B < 1 || s->H_q < 1 || s->H_kv < 1 || s->max_blocks < 1 || s->H_q % s->H_kv != 0) return LILY_ERR_INVALID;
    if (s->H_q / s->H_kv > kAttnMaxGroup || attn_stages(s->D, s->block_size) == 0) return LILY_ERR_UNSUPPORTED;
    return LILY_OK;
}

// Splits per (sequence, KV head): about one CTA per SM in all, at most one per
// cache block of the longest sequence.
int attn_splits(const lily_attn_shape &s, int sms)
{
    const int per = static_cast<int>(ceil_div(sms, static_cast<int64_t>(s.B) * s.H_kv));
    return std::max(1, std::min({per, s.max_blocks, kAttnMaxSplits}));
}

// Workspace: control block, then the partials of every (sequence, KV head,
// split) for up to kAttnMaxSplits splits (or max_blocks, if fewer).
struct AttnLayout {
    size_t ctrl, part_ml, part_acc, total;
};

AttnLayout attn_layout(const lily_attn_shape &s)
{
    const int64_t S = std::min(s.max_blocks, kAttnMaxSplits);
    const int64_t units = static_cast<int64_t>(s.B) * s.H_kv * S * kAttnMaxGroup;
    AttnLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + std::max<size_t>(bytes, 1));
        return at;
    };
    L.ctrl = take(sizeof(Ctrl));
    L.part_ml = take(units * 2 * 4);
    L.part_acc = take(units * s.D * 4);
    L.total = off;
    return L;
}

template <typename P>
P *at(void *ws, size_t off)
{
    return reinterpret_cast<P *>(static_cast<uint8_t *>(ws) + off);
}

// ------------------------------------------------------------------ validation
int check_shape(const lily_moe_shape *s)
{
    if (!s) return LILY_ERR_INVALID;
    if (s->T < 0 || s->d <= 0 || s->E <= 0 || s->top_k <= 0 || s->I <= 0 || s->I_shared <= 0 || s->group <= 0 ||
        s->block_rows <= 0)
        return LILY_ERR_INVALID;
    if (s->E != 256 || s->top_k != 8 || s->group != 64) return LILY_ERR_UNSUPPORTED;
    if (s->d % 256 != 0 || s->d > 16384) return LILY_ERR_UNSUPPORTED;
    if (s->I % 128 != 0 || s->I > 4096) return LILY_ERR_UNSUPPORTED;
    if (s->I_shared != s->I) return LILY_ERR_UNSUPPORTED;
    if (s->block_rows != 16 && s->block_rows != 32 && s->block_rows != 64 && s->block_rows != 128)
        return LILY_ERR_UNSUPPORTED;
    if (s->T > (1 << 20)) return LILY_ERR_UNSUPPORTED;
    return LILY_OK;
}

int check_q4(const lily_q4 &m)
{
    if (!m.q || !m.scale || !m.bias) return LILY_ERR_INVALID;
    if (!aligned16(m.q) || !aligned16(m.scale) || !aligned16(m.bias)) return LILY_ERR_MISALIGNED;
    return LILY_OK;
}

int check_weights(const lily_moe_weights *w)
{
    if (!w || !w->router_w) return LILY_ERR_INVALID;
    if (!aligned16(w->router_w) || (w->router_bias && !aligned16(w->router_bias))) return LILY_ERR_MISALIGNED;
    for (const lily_q4 *m : {&w->gate, &w->up, &w->down, &w->sh_gate, &w->sh_up, &w->sh_down}) {
        const int rc = check_q4(*m);
        if (rc) return rc;
    }
    return LILY_OK;
}

int check_ptr(const void *p)
{
    if (!p) return LILY_ERR_INVALID;
    if (!aligned16(p)) return LILY_ERR_MISALIGNED;
    return LILY_OK;
}

int check_ws(const void *ws, size_t ws_bytes, size_t need)
{
    const int rc = check_ptr(ws);
    if (rc) return rc;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return LILY_ERR_MISALIGNED;
    if (ws_bytes < need) return LILY_ERR_WORKSPACE;
    return LILY_OK;
}

// ------------------------------------------------------------------ device properties
int num_sms_current()
{
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
    return n;
}

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major tensor [rows][inner] with a box of [box_rows][box_inner].
bool make_tmap(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int elem_bytes, uint64_t inner, uint64_t rows,
               uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, std::max<uint64_t>(rows, 1)};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_bf16_sw128(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows)
{
    return make_tmap(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_f16_sw128(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows)
{
    return make_tmap(m, ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, inner, rows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed int4 rows: a box of 128 bytes (four k-steps of 64 weights) x 128 rows
// with the 128-byte swizzle, so the dequantisers read it without bank
// conflicts; boxes past the end of a row read zeros.
bool tmap_q4(CUtensorMap *m, const uint8_t *q, uint64_t K, uint64_t rows)
{
    return make_tmap(m, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

namespace {

// Token rows per router GEMM unit: 64 keeps more SMs busy than 128 at the
// prefill sizes (T = 8192 gives 128 units) at a small loss of MMA width.

// ------------------------------------------------------------------ enqueue helpers
// inv: where the scatter also writes the inverse permutation (NULL: not written).
// part: router_part_bytes(s) of scratch for the router's partial logits
// (router_ksplit(s) splits of K; unused when that is 1).
cudaError_t enqueue_route(const lily_moe_shape &s, const lily_moe_weights &w, const uint16_t *x,
                          const lily_moe_routing &r, float *logits, void *ws, float *part, cudaStream_t stream,
                          cudaEvent_t *events = nullptr, int *inv = nullptr)
{
    const PrefillLayout L = prefill_layout(s);
    Ctrl *ctrl = at<Ctrl>(ws, L.ctrl);
    CUtensorMap tmX, tmWr;
    if (!tmap_bf16_sw128(&tmX, x, s.d, s.T) || !tmap_bf16_sw128(&tmWr, w.router_w, s.d, s.E))
        return cudaErrorInvalidValue;

    GemmArgs g{};
    g.mode = kModeRouter;
    g.KT = gemm_k_steps(s.d);
    g.T = s.T; g.d = s.d; g.E = s.E; g.top_k = s.top_k; g.I = s.I;
    g.bm = kRouterBlockRows;
    g.K = s.d;
    g.m_tiles = 1;
    g.n_shared_blocks = static_cast<int>(ceil_div(s.T, kRouterBlockRows));
    g.n_routed_max = 0;
    g.router_bias = w.router_bias;
    g.logits = logits;
    g.ctrl = ctrl;
    const int sms = num_sms_current();
    const int ksplit = router_ksplit(s);
    g.ksplit = ksplit;
    g.logits_part = ksplit > 1 ? part : nullptr;
    const int grid = std::max(1, std::min(sms, g.n_shared_blocks * ksplit));
    cudaError_t e = launch_grouped_gemm(g, tmX, tmWr, tmWr, tmWr, tmWr, grid, stream);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[1], stream)) != cudaSuccess) return e;

    RouteArgs ra{};
    ra.T = s.T; ra.E = s.E; ra.top_k = s.top_k; ra.bm = s.block_rows;
    ra.logits = logits;
    ra.ksplit = ksplit;
    ra.logits_part = g.logits_part;
    ra.router_bias = w.router_bias;
    ra.topk_idx = r.topk_idx; ra.topk_w = r.topk_w;
    ra.counts = r.counts; ra.offsets = r.offsets; ra.perm = r.perm;
    ra.block_map = r.block_map; ra.n_blocks = r.n_blocks;
    ra.inv = inv;
    ra.chunk_counts = at<int>(ws, L.chunk_counts);
    ra.chunk_base = at<int>(ws, L.chunk_base);
    ra.n_chunks = static_cast<int>(route_chunks(s.T));
    ra.ctrl = ctrl;
    if (ra.n_chunks <= kRouteFusedChunks) {
        if ((e = launch_route_fused(ra, stream)) != cudaSuccess) return e;
    } else {
        if ((e = launch_topk_count(ra, stream)) != cudaSuccess) return e;
        if ((e = launch_route_scan(ra, stream)) != cudaSuccess) return e;
        if ((e = launch_scatter(ra, stream)) != cudaSuccess) return e;
    }
    if (events && (e = cudaEventRecord(events[2], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

// inv_ready: this workspace already holds the inverse of r.perm (the routing
// kernels of the same call wrote it).
cudaError_t enqueue_experts(const lily_moe_shape &s, const lily_moe_weights &w, const uint16_t *x,
                            const lily_moe_routing &r, float *out, void *ws, cudaStream_t stream,
                            cudaEvent_t *events, bool inv_ready)
{
    const PrefillLayout L = prefill_layout(s);
    Ctrl *ctrl = at<Ctrl>(ws, L.ctrl);
    __half *h = at<__half>(ws, L.h);
    __half *xs = at<__half>(ws, L.xs);
    int *inv = at<int>(ws, L.inv);
    const int64_t hrows = static_cast<int64_t>(s.top_k + 1) * s.T;
    CUtensorMap tmXs, tmH, tmG, tmU, tmD, tmSG, tmSU, tmSD;
    if (!tmap_f16_sw128(&tmXs, xs, s.d, hrows) || !tmap_f16_sw128(&tmH, h, s.I, hrows) ||
        !tmap_q4(&tmG, w.gate.q, s.d, static_cast<uint64_t>(s.E) * s.I) ||
        !tmap_q4(&tmU, w.up.q, s.d, static_cast<uint64_t>(s.E) * s.I) ||
        !tmap_q4(&tmD, w.down.q, s.I, static_cast<uint64_t>(s.E) * s.d) || !tmap_q4(&tmSG, w.sh_gate.q, s.d, s.I) ||
        !tmap_q4(&tmSU, w.sh_up.q, s.d, s.I) || !tmap_q4(&tmSD, w.sh_down.q, s.I, s.d))
        return cudaErrorInvalidValue;

    cudaError_t e = cudaSuccess;
    if (!inv_ready && (e = launch_invert_perm(r.perm, inv, s.T * s.top_k, &ctrl->status, stream)) != cudaSuccess) return e;
    if ((e = launch_prep_experts(x, inv, xs, s.T, s.d, s.top_k, &ctrl->status, stream)) != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[3], stream)) != cudaSuccess) return e;

    const int sms = num_sms_current();
    const int64_t cap = block_capacity(s);
    GemmArgs g{};
    g.T = s.T; g.d = s.d; g.E = s.E; g.top_k = s.top_k; g.I = s.I;
    g.bm = s.block_rows;
    g.n_shared_blocks = static_cast<int>(ceil_div(s.T, s.block_rows));
    g.n_routed_max = static_cast<int>(cap);
    g.n_blocks = r.n_blocks;
    g.block_map = r.block_map;
    g.perm = r.perm;
    g.topk_w = r.topk_w;
    g.xs = xs;
    g.h = h;
    g.out = out;
    g.ctrl = ctrl;

    g.ksplit = 1;
    // gate/up + SwiGLU
    g.mode = kModeGateUp;
    g.K = s.d;
    g.KT = gemm_k_steps(s.d);
    g.m_tiles = s.I / 128;
    g.s0 = w.gate.scale; g.b0 = w.gate.bias; g.s1 = w.up.scale; g.b1 = w.up.bias;
    g.ss0 = w.sh_gate.scale; g.sb0 = w.sh_gate.bias; g.ss1 = w.sh_up.scale; g.sb1 = w.sh_up.bias;
    int64_t units = (cap + g.n_shared_blocks) * g.m_tiles;
    int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms, units)));
    if ((e = launch_grouped_gemm(g, tmXs, tmG, tmU, tmSG, tmSU, grid, stream)) != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[4], stream)) != cudaSuccess) return e;

    // down + weighted combine
    g.mode = kModeDown;
    g.K = s.I;
    g.KT = gemm_k_steps(s.I);
    g.m_tiles = s.d / 256;
    g.s0 = g.s1 = w.down.scale; g.b0 = g.b1 = w.down.bias;
    g.ss0 = g.ss1 = w.sh_down.scale; g.sb0 = g.sb1 = w.sh_down.bias;
    units = (cap + g.n_shared_blocks) * g.m_tiles;
    grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms, units)));
    if ((e = launch_grouped_gemm(g, tmH, tmD, tmD, tmSD, tmSD, grid, stream)) != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[5], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

int check_routing(const lily_moe_routing *r, bool for_route)
{
    if (!r) return LILY_ERR_INVALID;
    int rc;
    if ((rc = check_ptr(r->topk_w)) || (rc = check_ptr(r->perm)) || (rc = check_ptr(r->block_map)) ||
        (rc = check_ptr(r->n_blocks)))
        return rc;
    if (for_route) {
        if ((rc = check_ptr(r->topk_idx)) || (rc = check_ptr(r->counts)) || (rc = check_ptr(r->offsets))) return rc;
        if (r->logits && !aligned16(r->logits)) return LILY_ERR_MISALIGNED;
    }
    return LILY_OK;
}

lily_moe_routing internal_routing(const lily_moe_shape &s, void *ws)
{
    const PrefillLayout L = prefill_layout(s);
    lily_moe_routing r{};
    r.logits = at<float>(ws, L.logits);
    r.topk_idx = at<int32_t>(ws, L.idx);
    r.topk_w = at<float>(ws, L.w);
    r.counts = at<int32_t>(ws, L.counts);
    r.offsets = at<int32_t>(ws, L.offsets);
    r.perm = at<int32_t>(ws, L.perm);
    r.block_map = at<int32_t>(ws, L.block_map);
    r.n_blocks = at<int32_t>(ws, L.n_blocks);
    return r;
}

// Text of the CUDA error behind this thread's last LILY_ERR_LAUNCH.
thread_local std::string t_last_error;

int cuda_fail(cudaError_t e, const char *what)
{
    t_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return LILY_ERR_LAUNCH;
}

int to_status(cudaError_t e, const char *what = "launch")
{
    return e == cudaSuccess ? LILY_OK : cuda_fail(e, what);
}

// ------------------------------------------------------------------ decode graph cache
struct GraphCache {
    std::mutex mu;
    std::unordered_map<std::string, cudaGraphExec_t> execs;
};
GraphCache &graph_cache()
{
    static GraphCache *c = new GraphCache();  // never destroyed: graphs live until process exit
    return *c;
}

}  // namespace

// Fixed scratch of lily_moe_route_noalloc.  Every GPU that loads the library
// holds it until the process exits.  In host code `g_noalloc_scratch` is only a
// host-side stand-in: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LILY_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch in the current context, looked up once
// per context (with its device current).  Returns nullptr if the lookup fails.
void *noalloc_scratch_address()
{
    static std::mutex mu;
    static std::unordered_map<unsigned long long, void *> addr;  // context id -> address
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (id != 0) {
        auto it = addr.find(id);
        if (it != addr.end()) return it->second;
    }
    // the lookup makes the device's primary context current if none was yet
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    const unsigned long long id2 = current_context_id();
    if (id2 != 0) addr[id2] = p;
    return p;
}

}  // namespace

extern "C" {

int lily_moe_version(void) { return kVersion; }

const char *lily_moe_status_string(int status)
{
    switch (status) {
    case LILY_OK: return "ok";
    case LILY_ERR_INVALID: return "invalid argument";
    case LILY_ERR_UNSUPPORTED: return "unsupported shape";
    case LILY_ERR_MISALIGNED: return "misaligned device pointer (16 bytes required; workspace 256 bytes)";
    case LILY_ERR_WORKSPACE: return "workspace too small";
    case LILY_ERR_LAUNCH: return "CUDA error while enqueueing";
    case LILY_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case LILY_ERR_DEVICE_INDEX: return "device index out of range";
    case LILY_ERR_SCRATCH_LIMIT: return "token count above the fixed scratch of lily_moe_route_noalloc";
    case LILY_ERR_DEVICE_RANGE: return "a value of x or h beyond the fp16 range of the expert GEMMs";
    default: return "unknown status";
    }
}

const char *lily_moe_last_error_detail(void) { return t_last_error.c_str(); }

int lily_moe_check_shape(const lily_moe_shape *shape) { return check_shape(shape); }

int64_t lily_moe_block_capacity(const lily_moe_shape *shape)
{
    if (check_shape(shape) != LILY_OK) return 0;
    return block_capacity(*shape);
}

size_t lily_moe_workspace_bytes(const lily_moe_shape *shape, int32_t n_layers_decode)
{
    if (check_shape(shape) != LILY_OK) return 0;
    size_t need = prefill_layout(*shape).total;
    if (n_layers_decode > 0) {
        if (shape->T < 1 || shape->T > 8 || shape->d > 4096 || shape->I > 1024) return 0;
        need = std::max(need, decode_layout(*shape).total);
    }
    return need;
}

int lily_moe_route(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x, lily_moe_routing *r,
                   void *ws, size_t ws_bytes, cudaStream_t stream)
{
    int rc;
    if ((rc = check_shape(shape)) || (rc = check_weights(w)) || (rc = check_routing(r, true))) return rc;
    if ((rc = check_ws(ws, ws_bytes, prefill_layout(*shape).total))) return rc;
    if (shape->T == 0) return LILY_OK;
    if ((rc = check_ptr(x))) return rc;
    float *logits = r->logits ? r->logits : at<float>(ws, prefill_layout(*shape).logits);
    const PrefillLayout L = prefill_layout(*shape);
    return to_status(enqueue_route(*shape, *w, x, *r, logits, ws, at<float>(ws, L.xs), stream, nullptr, at<int>(ws, L.inv)),
                     "routing launch");
}

int lily_moe_grouped_gemm(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                          const lily_moe_routing *r, float *out, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    int rc;
    if ((rc = check_shape(shape)) || (rc = check_weights(w)) || (rc = check_routing(r, false))) return rc;
    if ((rc = check_ws(ws, ws_bytes, prefill_layout(*shape).total))) return rc;
    if (shape->T == 0) return LILY_OK;
    if ((rc = check_ptr(x)) || (rc = check_ptr(out))) return rc;
    return to_status(enqueue_experts(*shape, *w, x, *r, out, ws, stream, nullptr, false), "expert launch");
}

int lily_moe_forward_timed(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x, float *out,
                           lily_moe_routing *r, void *ws, size_t ws_bytes, cudaStream_t stream, cudaEvent_t *events)
{
    int rc;
    if ((rc = check_shape(shape)) || (rc = check_weights(w))) return rc;
    if (r && (rc = check_routing(r, true))) return rc;
    if ((rc = check_ws(ws, ws_bytes, prefill_layout(*shape).total))) return rc;
    if (shape->T == 0) return LILY_OK;
    if ((rc = check_ptr(x)) || (rc = check_ptr(out))) return rc;
    const lily_moe_routing rr = r ? *r : internal_routing(*shape, ws);
    float *logits = rr.logits ? rr.logits : at<float>(ws, prefill_layout(*shape).logits);
    cudaError_t e;
    if (events && (e = cudaEventRecord(events[0], stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    const PrefillLayout L = prefill_layout(*shape);
    if ((e = enqueue_route(*shape, *w, x, rr, logits, ws, at<float>(ws, L.xs), stream, events, at<int>(ws, L.inv))) !=
        cudaSuccess)
        return cuda_fail(e, "routing launch");
    return to_status(enqueue_experts(*shape, *w, x, rr, out, ws, stream, events, true), "expert launch");
}

int lily_moe_forward(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x, float *out,
                     lily_moe_routing *r, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return lily_moe_forward_timed(shape, w, x, out, r, ws, ws_bytes, stream, nullptr);
}

int lily_moe_decode(const lily_moe_shape *shape, int32_t n_layers, const lily_moe_weights *layers, const uint16_t *x,
                    float *out, uint16_t *x_next, const lily_moe_decode_trace *trace, void *ws, size_t ws_bytes,
                    cudaStream_t stream)
{
    int rc;
    if ((rc = check_shape(shape))) return rc;
    if (n_layers < 1 || !layers) return LILY_ERR_INVALID;
    if (shape->T < 1 || shape->T > 8 || shape->d > 4096 || shape->I > 1024) return LILY_ERR_UNSUPPORTED;
    for (int l = 0; l < n_layers; ++l)
        if ((rc = check_weights(&layers[l]))) return rc;
    if ((rc = check_ws(ws, ws_bytes, decode_layout(*shape).total))) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(out))) return rc;
    if (x_next && !aligned16(x_next)) return LILY_ERR_MISALIGNED;
    if (trace && ((trace->logits && !aligned16(trace->logits)) || (trace->topk_idx && !aligned16(trace->topk_idx)) ||
                  (trace->topk_w && !aligned16(trace->topk_w))))
        return LILY_ERR_MISALIGNED;

    const lily_moe_shape s = *shape;
    const DecodeLayout L = decode_layout(s);
    const int sms = num_sms_current();
    const size_t td = static_cast<size_t>(s.T) * s.d;

    auto enqueue_all = [&](cudaStream_t st) -> cudaError_t {
        Ctrl *ctrl = at<Ctrl>(ws, L.ctrl);
        cudaError_t e = cudaMemsetAsync(&ctrl->ticket2, 0, sizeof(unsigned int), st);
        if (e != cudaSuccess) return e;
        for (int l = 0; l < n_layers; ++l) {
            const lily_moe_weights &w = layers[l];
            DecodeLayerArgs a{};
            a.T = s.T; a.d = s.d; a.E = s.E; a.top_k = s.top_k; a.I = s.I; a.layer = l;
            a.router_w = w.router_w; a.router_bias = w.router_bias;
            a.gate_q = w.gate.q; a.up_q = w.up.q; a.down_q = w.down.q;
            a.gate_s = w.gate.scale; a.gate_b = w.gate.bias; a.up_s = w.up.scale; a.up_b = w.up.bias;
            a.down_s = w.down.scale; a.down_b = w.down.bias;
            a.sh_gate_q = w.sh_gate.q; a.sh_up_q = w.sh_up.q; a.sh_down_q = w.sh_down.q;
            a.sh_gate_s = w.sh_gate.scale; a.sh_gate_b = w.sh_gate.bias; a.sh_up_s = w.sh_up.scale;
            a.sh_up_b = w.sh_up.bias; a.sh_down_s = w.sh_down.scale; a.sh_down_b = w.sh_down.bias;
            a.x_in = l == 0 ? x : nullptr;
            a.prev_out = l == 0 ? nullptr : out + (l - 1) * td;
            a.out = out + l * td;
            a.x_export = (l > 0 && x_next) ? x_next + (l - 1) * td : nullptr;
            if (trace) {
                a.trace_logits = trace->logits ? trace->logits + static_cast<size_t>(l) * s.T * s.E : nullptr;
                a.trace_idx = trace->topk_idx ? trace->topk_idx + static_cast<size_t>(l) * s.T * s.top_k : nullptr;
                a.trace_w = trace->topk_w ? trace->topk_w + static_cast<size_t>(l) * s.T * s.top_k : nullptr;
            }
            a.x_cur = at<uint16_t>(ws, L.x_cur);
            a.xp = at<__half>(ws, L.xp);
            a.logits = at<float>(ws, L.logits);
            a.n_units = at<int>(ws, L.n_units);
            a.unit_expert = at<int>(ws, L.unit_expert);
            a.unit_mask = at<int>(ws, L.unit_mask);
            a.unit_w = at<float>(ws, L.unit_w);
            a.h = at<__half>(ws, L.h);
            a.ctrl = ctrl;
            if ((e = launch_decode_layer(a, sms, st)) != cudaSuccess) return e;
        }
        if (x_next)
            return launch_decode_final_norm(out + (n_layers - 1) * td, x_next + (n_layers - 1) * td, s.T, s.d, st);
        return cudaSuccess;
    };

    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone) return to_status(enqueue_all(stream), "decode launch (capturing stream)");

    // Key: every argument value that the recorded launches depend on.
    std::string key;
    auto put = [&key](const void *p, size_t n) { key.append(static_cast<const char *>(p), n); };
    int dev = 0;
    cudaGetDevice(&dev);
    put(&dev, sizeof dev);
    // the context the graph was instantiated in (a reset device gets a new one)
    const unsigned long long ctx_id = current_context_id();
    put(&ctx_id, sizeof ctx_id);
    put(&s, sizeof s);
    put(&n_layers, sizeof n_layers);
    put(layers, sizeof(lily_moe_weights) * n_layers);
    put(&x, sizeof x); put(&out, sizeof out); put(&x_next, sizeof x_next); put(&ws, sizeof ws);
    const lily_moe_decode_trace tr = trace ? *trace : lily_moe_decode_trace{};
    put(&tr, sizeof tr);

    GraphCache &gc = graph_cache();
    std::lock_guard<std::mutex> lock(gc.mu);
    auto it = gc.execs.find(key);
    if (it == gc.execs.end()) {
        cudaStream_t cap;
        if ((ce = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(ce, "cudaStreamCreateWithFlags");
        cudaGraph_t graph = nullptr;
        cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
        if (e == cudaSuccess) {
            const cudaError_t e1 = enqueue_all(cap);
            const cudaError_t e2 = cudaStreamEndCapture(cap, &graph);
            e = e1 != cudaSuccess ? e1 : e2;
        }
        cudaGraphExec_t exec = nullptr;
        if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        cudaStreamDestroy(cap);
        if (e != cudaSuccess) return cuda_fail(e, "decode graph capture / instantiate");
        if (gc.execs.size() >= 64) {
            for (auto &kv : gc.execs) cudaGraphExecDestroy(kv.second);
            gc.execs.clear();
        }
        it = gc.execs.emplace(key, exec).first;
    }
    return to_status(cudaGraphLaunch(it->second, stream), "cudaGraphLaunch (decode)");
}

size_t lily_attn_workspace_bytes(const lily_attn_shape *shape)
{
    if (attn_check_shape(shape) != LILY_OK) return 0;
    return attn_layout(*shape).total;
}

int lily_attn_decode(const lily_attn_shape *shape, const uint16_t *q, const uint16_t *k_cache,
                     const uint16_t *v_cache, int64_t n_cache_blocks, const int32_t *block_table,
                     const int32_t *seq_lens, float scale, float *out, void *ws, size_t ws_bytes,
                     cudaStream_t stream)
{
    int rc;
    if ((rc = attn_check_shape(shape))) return rc;
    const lily_attn_shape s = *shape;
    if (n_cache_blocks < 1 || !std::isfinite(scale)) return LILY_ERR_INVALID;
    if (n_cache_blocks * s.H_kv * s.block_size >= (int64_t(1) << 31)) return LILY_ERR_UNSUPPORTED;
    const AttnLayout L = attn_layout(s);
    if ((rc = check_ws(ws, ws_bytes, L.total))) return rc;
    for (const void *p : {static_cast<const void *>(q), static_cast<const void *>(k_cache),
                          static_cast<const void *>(v_cache), static_cast<const void *>(block_table),
                          static_cast<const void *>(seq_lens), static_cast<const void *>(out)})
        if ((rc = check_ptr(p))) return rc;
    const uint64_t rows = static_cast<uint64_t>(n_cache_blocks) * s.H_kv * s.block_size;
    CUtensorMap tmK, tmV;
    if (!make_tmap(&tmK, k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.D, rows, 64, s.block_size,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&tmV, v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.D, rows, 64, s.block_size,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (KV cache)");
    AttnArgs a{};
    a.B = s.B; a.H_q = s.H_q; a.H_kv = s.H_kv; a.D = s.D; a.bs = s.block_size; a.max_blocks = s.max_blocks;
    a.group = s.H_q / s.H_kv;
    a.n_splits = attn_splits(s, num_sms_current());
    a.n_cache_blocks = n_cache_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.q = q;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.part_ml = at<float>(ws, L.part_ml);
    a.part_acc = at<float>(ws, L.part_acc);
    a.out = out;
    a.ctrl = at<Ctrl>(ws, L.ctrl);
    return to_status(launch_attn_decode(a, tmK, tmV, stream), "attention launch");
}

int lily_gdn_scan(const lily_gdn_shape *shape, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *alpha, const float *beta, const float *state_in, float scale, float *out,
                  float *state_out, cudaStream_t stream)
{
    if (!shape) return LILY_ERR_INVALID;
    const lily_gdn_shape s = *shape;
    if (s.T < 0 || s.H_k < 1 || s.H_v < 1 || s.H_v % s.H_k != 0 || !std::isfinite(scale)) return LILY_ERR_INVALID;
    if ((s.d_k != 64 && s.d_k != 128) || s.d_v < 16 || s.d_v > 1024 || s.d_v % 16 != 0) return LILY_ERR_UNSUPPORTED;
    int rc;
    // with T = 0 the token arrays are empty and may be NULL
    if (s.T > 0)
        for (const void *p : {static_cast<const void *>(q), static_cast<const void *>(k), static_cast<const void *>(v),
                              static_cast<const void *>(alpha), static_cast<const void *>(beta),
                              static_cast<const void *>(out)})
            if ((rc = check_ptr(p))) return rc;
    if ((rc = check_ptr(state_out))) return rc;
    if (state_in && !aligned16(state_in)) return LILY_ERR_MISALIGNED;
    if (state_in == state_out) return LILY_ERR_INVALID;
    GdnArgs a{};
    a.T = s.T; a.H_k = s.H_k; a.H_v = s.H_v; a.d_k = s.d_k; a.d_v = s.d_v;
    a.scale = scale;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
    a.state_in = state_in; a.out = out; a.state_out = state_out;
    return to_status(launch_gdn_scan(a, stream), "Gated DeltaNet scan launch");
}

int lily_moe_route_noalloc(const lily_moe_shape *shape, const lily_moe_weights *w, const uint16_t *x,
                           lily_moe_routing *r, int32_t *device_status, cudaStream_t stream)
{
    int rc;
    if ((rc = check_shape(shape)) || (rc = check_weights(w)) || (rc = check_routing(r, true))) return rc;
    if (shape->T > LILY_NOALLOC_MAX_TOKENS) return LILY_ERR_SCRATCH_LIMIT;
    if ((rc = check_ptr(r->logits))) return rc;
    if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return LILY_ERR_MISALIGNED;
    // The routing kernels touch only the control block and the two per-chunk
    // tables of the prefill workspace layout, then the router's partial logits
    // (placed after the tables here), which fit in the fixed scratch.
    const PrefillLayout L = prefill_layout(*shape);
    const size_t part_off =
        align_up(L.chunk_base + static_cast<size_t>(route_chunks(shape->T)) * shape->E * 4);
    if (part_off + router_part_bytes(*shape) > LILY_NOALLOC_SCRATCH_BYTES) return LILY_ERR_SCRATCH_LIMIT;
    if (shape->T == 0) {
        // nothing to route; the call's status (OK) still goes to device_status
        cudaError_t e;
        if (device_status && (e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), stream)) != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync (device_status)");
        return LILY_OK;
    }
    if ((rc = check_ptr(x))) return rc;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return cuda_fail(cudaGetLastError(), "cudaGetSymbolAddress (fixed scratch)");
    // The scratch keeps the previous call's contents: start from a clear control block.
    cudaError_t e;
    if ((e = cudaMemsetAsync(scratch, 0, sizeof(Ctrl), stream)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    if ((e = enqueue_route(*shape, *w, x, *r, r->logits, scratch, at<float>(scratch, part_off), stream)) != cudaSuccess)
        return cuda_fail(e, "routing launch");
    if (device_status &&
        (e = cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync (device_status)");
    return LILY_OK;
}

int lily_moe_device_status(const void *ws, cudaStream_t stream)
{
    if (!ws) return LILY_ERR_INVALID;
    cudaError_t e;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int status = 0;
    if ((e = cudaMemcpy(&status, ws, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy (status word)");
    return status;
}

int lily_moe_clear_status(void *ws, cudaStream_t stream)
{
    if (!ws) return LILY_ERR_INVALID;
    return to_status(cudaMemsetAsync(ws, 0, sizeof(int), stream), "cudaMemsetAsync (status word)");
}

}  // extern "C"
