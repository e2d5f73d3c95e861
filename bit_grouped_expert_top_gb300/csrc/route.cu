// Routing tables of the MoE layer, kept entirely on the GPU.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br): a router scores 256
// experts and picks eight (section "O modelo em tres formatos de carga"); the
// routing histogram, prefix scan, scatter and block map stay inside one GPU
// submission with no CPU synchronisation (section "Prefill e decode").
//
// Three kernels, one stream, no host sync (for at most kRouteFusedChunks
// chunks the three steps run as one kernel, route_fused_kernel, with a grid
// barrier between the counts and the scatter):
//   topk_count_kernel : (when the router split K: adds the partial logits in
//                       split order and the bias, and writes the logits) one
//                       warp per token selects the top 8 of 256 fp32 logits
//                       (descending; lower index first among equal logits) in
//                       eight warp-maximum rounds and computes the renormalised
//                       softmax weights; each CTA then counts its chunk of
//                       tokens per expert (32 tokens; 8 or 16 for small T).
//   scan_kernel       : one CTA per expert scans that expert's per-chunk counts
//                       in chunk order (each chunk's base within the expert) and
//                       writes its total; the last CTA to finish (ticket
//                       counter) scans the totals over experts into offsets and
//                       writes the block map.
//   scatter_kernel    : each CTA writes its chunk's assignments into
//                       expert-sorted order; ranks inside the chunk come from
//                       __match_any_sync plus per-warp counts, so the order
//                       within an expert is ascending (token, slot) and the
//                       result is deterministic (no atomics decide positions).
#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kRouteThreads = 256;               // 8 warps
constexpr int kE = 256;                          // experts (one per thread in the scans)
constexpr int kTopK = 8;

__device__ __forceinline__ unsigned int ld_acquire_gpu_u32(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Exclusive scan over the 256 threads of the block; returns the exclusive
// prefix, writes the total to *total.
__device__ __forceinline__ int block_exclusive_scan_256(int v, int *scratch /* [8] */, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int warp_off = 0, sum = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int s = scratch[w];
        if (w < warp) warp_off += s;
        sum += s;
    }
    __syncthreads();
    *total = sum;
    return warp_off + incl - v;
}

// Top-8 and weights of the chunk's CT tokens and the chunk's per-expert counts
// (into hist, zeroed and complete on return).  SPLIT: the router split K
// (a.ksplit > 1 partial sums, no bias).
template <bool SPLIT, int CT>
__device__ __forceinline__ void topk_chunk(const RouteArgs &a, int chunk, int *hist)
{
    constexpr int kTokPerWarp = CT / 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    hist[threadIdx.x] = 0;
    __syncthreads();

    // each warp's tokens, the next token's logits (or partial logits) loaded
    // while this one is ranked; lane l holds experts 8 l .. 8 l + 7
    const int t0 = chunk * CT + warp * kTokPerWarp;
    const int S = SPLIT ? a.ksplit : 1;
    constexpr int NS = SPLIT ? kMaxRouterSplit : 1;
    float4 bias0 = make_float4(0.f, 0.f, 0.f, 0.f), bias1 = bias0;
    if (SPLIT && a.router_bias) {
        bias0 = *reinterpret_cast<const float4 *>(a.router_bias + lane * 8);
        bias1 = *reinterpret_cast<const float4 *>(a.router_bias + lane * 8 + 4);
    }
    float4 n0[NS], n1[NS];
    auto load_next = [&](int t) {
        const float *base = SPLIT ? a.logits_part : a.logits;
#pragma unroll
        for (int s2 = 0; s2 < NS; ++s2) {
            if (s2 < S) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    base + (static_cast<size_t>(s2) * a.T + t) * kE + lane * 8);
                n0[s2] = __ldcg(src);
                n1[s2] = __ldcg(src + 1);
            }
        }
    };
    if (t0 < a.T) load_next(t0);
    for (int i = 0; i < kTokPerWarp; ++i) {
        const int t = t0 + i;
        if (t >= a.T) break;
        float4 c0 = n0[0], c1 = n1[0];
        if (SPLIT) {
#pragma unroll
            for (int s2 = 1; s2 < NS; ++s2) {
                if (s2 < S) {
                    c0.x += n0[s2].x; c0.y += n0[s2].y; c0.z += n0[s2].z; c0.w += n0[s2].w;
                    c1.x += n1[s2].x; c1.y += n1[s2].y; c1.z += n1[s2].z; c1.w += n1[s2].w;
                }
            }
            c0.x += bias0.x; c0.y += bias0.y; c0.z += bias0.z; c0.w += bias0.w;
            c1.x += bias1.x; c1.y += bias1.y; c1.z += bias1.z; c1.w += bias1.w;
            float4 *dst = reinterpret_cast<float4 *>(a.logits + static_cast<size_t>(t) * kE + lane * 8);
            dst[0] = c0;
            dst[1] = c1;
        }
        const float lv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        if (i + 1 < kTokPerWarp && t + 1 < a.T) load_next(t + 1);
        int sel_e;
        float sel_w;
        warp_top8_keys(lv, lane, sel_e, sel_w);
        if (lane < kTopK) {
            a.topk_idx[static_cast<size_t>(t) * kTopK + lane] = sel_e;
            a.topk_w[static_cast<size_t>(t) * kTopK + lane] = sel_w;
            atomicAdd(&hist[sel_e], 1);
        }
    }
    __syncthreads();
}

template <bool SPLIT>
__global__ void __launch_bounds__(kRouteThreads)
topk_count_kernel(const RouteArgs a)
{
    __shared__ int hist[kE];
    pdl_trigger();
    pdl_wait();  // the router's logits are complete
    topk_chunk<SPLIT, kRouteChunkTokens>(a, blockIdx.x, hist);
    a.chunk_counts[static_cast<size_t>(blockIdx.x) * kE + threadIdx.x] = hist[threadIdx.x];
}

// CTA e: exclusive scan of expert e's per-chunk counts in chunk order (chunk
// bases relative to the expert's first sorted row) and the expert's total.
// The last CTA scans the totals over experts and writes the block map.
// Thread x = expert x with its total total_e: returns the expert's first row in
// expert-sorted order (exclusive scan over experts); if `write`, also writes
// counts-derived offsets, n_blocks and the block map.
__device__ __forceinline__ int expert_tables(const RouteArgs &a, int total_e, int *scratch, bool write)
{
    const int x = threadIdx.x;  // expert
    int sum_all;
    const int off = block_exclusive_scan_256(total_e, scratch, &sum_all);
    if (!write) return off;
    const int nb = (total_e + a.bm - 1) / a.bm;
    int nb_all;
    const int bstart = block_exclusive_scan_256(nb, scratch, &nb_all);
    a.offsets[x] = off;
    if (x == kE - 1) a.offsets[kE] = off + total_e;
    if (x == 0) *a.n_blocks = nb_all;
    for (int b = 0; b < nb; ++b) {
        int *ent = a.block_map + 3 * static_cast<size_t>(bstart + b);
        ent[0] = x;
        ent[1] = off + b * a.bm;
        ent[2] = min(a.bm, total_e - b * a.bm);
    }
    return off;
}

__global__ void __launch_bounds__(kRouteThreads)
scan_kernel(const RouteArgs a)
{
    __shared__ int scratch[8];
    __shared__ int is_last;
    const int e = blockIdx.x;
    int carry = 0;
    pdl_trigger();
    pdl_wait();  // the per-chunk counts are complete
    for (int c0 = 0; c0 < a.n_chunks; c0 += kRouteThreads) {
        const int c = c0 + threadIdx.x;
        const size_t i = static_cast<size_t>(c) * kE + e;
        const int v = c < a.n_chunks ? a.chunk_counts[i] : 0;
        int tile_total;
        const int ex = block_exclusive_scan_256(v, scratch, &tile_total);
        if (c < a.n_chunks) a.chunk_base[i] = carry + ex;
        carry += tile_total;
    }
    if (threadIdx.x == 0) a.counts[e] = carry;

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(&a.ctrl->ticket, 1u);
        is_last = (prev == static_cast<unsigned int>(gridDim.x) - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    expert_tables(a, __ldcg(a.counts + threadIdx.x), scratch, true);
    if (threadIdx.x == 0) a.ctrl->ticket = 0u;
}

// Writes the chunk's (CT tokens') assignments into expert-sorted order; base[e]
// (shared, set and visible on entry) is the chunk's first row of expert e.
template <int CT>
__device__ __forceinline__ void scatter_chunk(const RouteArgs &a, int chunk, int *base, int (*cnt)[kE])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int n_assign = CT * kTopK;  // assignments per chunk
    const int total = a.T * kTopK;
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int round = 0; round < (n_assign + kRouteThreads - 1) / kRouteThreads; ++round) {
        const int ga = chunk * n_assign + round * kRouteThreads + threadIdx.x;  // = t*8 + j
        const bool valid = round * kRouteThreads + static_cast<int>(threadIdx.x) < n_assign && ga < total;
        int e = valid ? a.topk_idx[ga] : -1;
        if (valid && (e < 0 || e >= kE)) {
            record_error(&a.ctrl->status, kErrDeviceIndex);
            e = -1;
        }
#pragma unroll
        for (int w = 0; w < 8; ++w) cnt[w][threadIdx.x] = 0;
        __syncthreads();
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt_mask);
        if (e >= 0 && rank == 0) cnt[warp][e] = __popc(same);
        __syncthreads();
        // per expert: exclusive prefix over the 8 warps
        int run = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const int c = cnt[w][threadIdx.x];
            cnt[w][threadIdx.x] = run;
            run += c;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = base[e] + cnt[warp][e] + rank;
            if (pos >= 0 && pos < total) {
                a.perm[pos] = ga;
                if (a.inv) a.inv[ga] = pos;
            } else {
                record_error(&a.ctrl->status, kErrDeviceIndex);
            }
        }
        __syncthreads();
        base[threadIdx.x] += run;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kRouteThreads)
scatter_kernel(const RouteArgs a)
{
    __shared__ int cnt[8][kE];
    __shared__ int base[kE];
    pdl_trigger();
    pdl_wait();  // offsets and chunk bases are complete
    base[threadIdx.x] = a.offsets[threadIdx.x] + a.chunk_base[static_cast<size_t>(blockIdx.x) * kE + threadIdx.x];
    __syncthreads();
    scatter_chunk<kRouteChunkTokens>(a, blockIdx.x, base, cnt);
}

// The three steps in one launch, for at most kRouteFusedChunks chunks (all CTAs
// resident): top-8 and counts per chunk; a grid barrier (arrival count in the
// control block, reset by the router GEMM of the same call); then every CTA
// adds up the chunk counts it needs (all chunks for the totals, the earlier
// ones for its own base), CTA 0 writes counts, offsets and the block map, and
// each CTA scatters its chunk.
template <bool SPLIT, int CT>
__global__ void __launch_bounds__(kRouteThreads)
route_fused_kernel(const RouteArgs a)
{
    __shared__ int hist[kE];
    __shared__ int cnt[8][kE];
    __shared__ int base[kE];
    __shared__ int scratch[8];
    __shared__ int go;
    const int chunk = blockIdx.x;
    pdl_trigger();
    pdl_wait();  // the router's logits (and its reset of the arrival count) are complete
    topk_chunk<SPLIT, CT>(a, chunk, hist);
    a.chunk_counts[static_cast<size_t>(chunk) * kE + threadIdx.x] = hist[threadIdx.x];
    __syncthreads();  // every count of this chunk stored
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(&a.ctrl->ticket, 1u);
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu_u32(&a.ctrl->ticket) < static_cast<unsigned int>(gridDim.x)) {
            if (global_timer_ns() - t0 > LILY_WAIT_LIMIT_NS) {
                record_error(&a.ctrl->status, kErrDeviceTimeout);
                ok = 0;
                break;
            }
        }
        __threadfence();
        go = ok;
    }
    __syncthreads();
    if (!go) return;
    int total_e = 0, prefix_e = 0;
#pragma unroll 8
    for (int c = 0; c < a.n_chunks; ++c) {
        const int v = __ldcg(a.chunk_counts + static_cast<size_t>(c) * kE + threadIdx.x);
        total_e += v;
        if (c < chunk) prefix_e += v;
    }
    if (chunk == 0) a.counts[threadIdx.x] = total_e;
    const int off = expert_tables(a, total_e, scratch, chunk == 0);
    base[threadIdx.x] = off + prefix_e;
    __syncthreads();
    scatter_chunk<CT>(a, chunk, base, cnt);
}

}  // namespace

cudaError_t launch_topk_count(const RouteArgs &a, cudaStream_t stream)
{
    if (a.ksplit > 1) return launch_pdl(topk_count_kernel<true>, dim3(a.n_chunks), dim3(kRouteThreads), 0, stream, a);
    return launch_pdl(topk_count_kernel<false>, dim3(a.n_chunks), dim3(kRouteThreads), 0, stream, a);
}

cudaError_t launch_route_fused(const RouteArgs &a, cudaStream_t stream)
{
    const dim3 grid(a.n_chunks), block(kRouteThreads);
    const bool split = a.ksplit > 1;
    switch (route_chunk_tokens(a.T)) {
    case 8:
        return split ? launch_pdl(route_fused_kernel<true, 8>, grid, block, 0, stream, a)
                     : launch_pdl(route_fused_kernel<false, 8>, grid, block, 0, stream, a);
    case 16:
        return split ? launch_pdl(route_fused_kernel<true, 16>, grid, block, 0, stream, a)
                     : launch_pdl(route_fused_kernel<false, 16>, grid, block, 0, stream, a);
    default:
        return split ? launch_pdl(route_fused_kernel<true, 32>, grid, block, 0, stream, a)
                     : launch_pdl(route_fused_kernel<false, 32>, grid, block, 0, stream, a);
    }
}

cudaError_t launch_route_scan(const RouteArgs &a, cudaStream_t stream)
{
    return launch_pdl(scan_kernel, dim3(kE), dim3(kRouteThreads), 0, stream, a);
}

cudaError_t launch_scatter(const RouteArgs &a, cudaStream_t stream)
{
    return launch_pdl(scatter_kernel, dim3(a.n_chunks), dim3(kRouteThreads), 0, stream, a);
}

}  // namespace lily
