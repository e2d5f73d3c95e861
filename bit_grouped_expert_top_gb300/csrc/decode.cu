// Decode path of the MoE layer for 1..8 tokens: fused dequant-GEMVs.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br, section "Prefill e
// decode: onde estao os ganhos"): at batch 1 there is almost no weight reuse,
// so memory bandwidth sets the ceiling.  Only the bytes of the selected
// experts (plus the shared expert and the router) are read, each exactly once,
// with 16-byte coalesced loads, dequantised in registers (weights rounded once
// to fp16, as in the prefill path) and accumulated in fp32.
//
// Three kernels per layer:
//   dec_route_kernel  : builds the layer input (layer 0: x; later layers: the
//                       parameter-free RMS norm of the previous output, rounded
//                       to bf16) and the router GEMV (one warp per expert).
//   dec_gateup_kernel : every CTA computes the top-8 selection per token from
//                       the logits and the list of distinct experts ("units")
//                       with per-token weights (the shared expert is unit 0
//                       with weight 1); then a tensor-core GEMV (mma.sync
//                       m16n8k16, the tokens as the 8 columns): per unit and 32
//                       rows of I, gate and up dequantised in registers, SwiGLU,
//                       scaled by the unit's routing weight per token, h' stored
//                       as fp16.
//   dec_down_kernel   : tensor-core GEMV over K = units x I: per 16 output
//                       rows, sum over the units of Wd h' (deterministic, no
//                       atomics).
#include <algorithm>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxT = 8;
// Read-only loads issued as volatile asm, so that the compiler keeps them where
// they are written (a plain read-only load may be moved past pdl_wait to its
// first use, which would undo a prefetch meant to overlap the previous grid).
__device__ __forceinline__ uint4 ld_early(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_early8(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_early_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// acc + dot of 8 bf16 weights with 8 bf16 activations (fp32).
__device__ __forceinline__ float dot8_bf16(uint4 w, uint4 x, float acc)
{
    const uint32_t wu[4] = {w.x, w.y, w.z, w.w}, xu[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wu[p]));
        const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xu[p]));
        acc = fmaf(wf.x, xf.x, acc);
        acc = fmaf(wf.y, xf.y, acc);
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- tensor-core GEMVs
// The expert GEMVs run on mma.sync m16n8k16 (f16 x f16 -> f32): 16 weight rows
// x 16 K x 8 token columns per instruction (tokens >= T are zero columns), so a
// weight is dequantised once for all tokens.  Lane (g = lane / 4, t = lane % 4)
// loads 16 bytes (32 weights) of rows g and g + 8 for each 128-wide K block:
// weights [32 t, 32 t + 32) of the block.  The K order inside the block is
// permuted so that these weights are exactly this lane's A-fragment entries:
// within 32-bit word w (weights 8w..8w+7, rebuilt in pairs (0,2) (4,6) (1,3)
// (5,7) by dequant8_f16_e2m3), weight e goes to slice 2w + (e & 1), entry e >> 1
// of the lane's four K positions.  The B operand
// (x, or h for the down projection) is stored in the same permuted order, so
// each lane reads its B fragment with one 8-byte load.
constexpr int kKB = 128;  // K block

// Position of element k (of a K range starting at 0) in the permuted B layout
// [kb][n][t][s][4] for token column n of 8.
__device__ __forceinline__ int perm_b_index(int k, int n)
{
    const int kb = k >> 7, r = k & 127, t = r >> 5, w = (r & 31) >> 3, e = r & 7;
    const int s = 2 * w + (e & 1), idx = e >> 1;
    return (((kb * 8 + n) * 4 + t) * 8 + s) * 4 + idx;
}

// KEEP: float4 of the previous output a thread may keep in registers (4 or 8;
// the smaller copy has less code to fetch when few values are kept).
template <int KEEP>
__global__ void __launch_bounds__(kDecThreads)
dec_route_kernel(const DecodeLayerArgs a)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(dsm);  // [T][d] plain layout
    __shared__ float red[kDecWarps][kMaxT];
    __shared__ float inv_rms[kMaxT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = a.T, d = a.d;
    const int e = blockIdx.x * kDecWarps + warp;  // this warp's expert
    const uint4 *wrow = reinterpret_cast<const uint4 *>(a.router_w + static_cast<size_t>(e < a.E ? e : 0) * d);
    const int n8 = d / 8;  // 16-byte chunks of a router row

    // The router row does not depend on the layer input: start its loads first.
    constexpr int kPre = 8;
    uint4 wpre[kPre];
#pragma unroll
    for (int m = 0; m < kPre; ++m) {
        const int c = lane + 32 * m;
        if (e < a.E && c < n8) wpre[m] = ld_early(wrow + c);
    }

    pdl_trigger();
    pdl_wait();  // the previous layer's output (and this call's buffers) are ready

    // ---- layer input
    if (a.prev_out == nullptr) {
        for (int i = threadIdx.x; i < T * d / 8; i += kDecThreads)
            reinterpret_cast<uint4 *>(xs)[i] = reinterpret_cast<const uint4 *>(a.x_in)[i];
    } else {
        // the sum of squares, then the scaled bf16 input; a thread's values are
        // kept in registers when they are at most KEEP float4 in all,
        // else read again in a second pass.  Each pass has all of a thread's
        // loads in flight at once (d <= 4096: at most 4 float4 per thread and token).
        const int d4 = d / 4;
        const int J = (d4 + kDecThreads - 1) / kDecThreads;  // float4 per thread and token
        const bool kept = T * J <= KEEP;
        const float4 *po = reinterpret_cast<const float4 *>(a.prev_out);
        float4 keep[KEEP];
        if (kept) {
#pragma unroll
            for (int q = 0; q < KEEP; ++q) {
                const int t = q / J, c = threadIdx.x + (q - t * J) * kDecThreads;
                keep[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < T && c < d4) keep[q] = __ldcg(po + static_cast<size_t>(t) * d4 + c);
            }
#pragma unroll
            for (int t = 0; t < KEEP; ++t) {
                if (t < T) {
                    float ss = 0.0f;
#pragma unroll
                    for (int q = 0; q < KEEP; ++q) {
                        if (q / J == t) {
                            const float4 v = keep[q];
                            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
                        }
                    }
                    ss = warp_sum(ss);
                    if (lane == 0) red[warp][t] = ss;
                }
            }
        } else {
#pragma unroll 4
            for (int t = 0; t < T; ++t) {  // up to four tokens' loads in flight together
                float ss = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = threadIdx.x + j * kDecThreads;
                    if (c < d4) {
                        const float4 v = __ldcg(po + static_cast<size_t>(t) * d4 + c);
                        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0) red[warp][t] = ss;
            }
        }
        __syncthreads();
        if (threadIdx.x < T) {
            float s = 0.0f;
            for (int w = 0; w < kDecWarps; ++w) s += red[w][threadIdx.x];
            inv_rms[threadIdx.x] = 1.0f / sqrtf(s / static_cast<float>(d) + 1e-6f);
        }
        __syncthreads();
        auto put = [&](int t, int c, float4 v) {
            const float r = inv_rms[t];
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r, v.y * r), hi = __floats2bfloat162_rn(v.z * r, v.w * r);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t *>(&lo);
            o.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(xs + static_cast<size_t>(t) * d + 4 * c) = o;
        };
        if (kept) {
#pragma unroll
            for (int q = 0; q < KEEP; ++q) {
                const int t = q / J, c = threadIdx.x + (q - t * J) * kDecThreads;
                if (t < T && c < d4) put(t, c, keep[q]);
            }
        } else {
#pragma unroll 4
            for (int t = 0; t < T; ++t) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = threadIdx.x + j * kDecThreads;
                    if (c < d4) put(t, c, __ldcg(po + static_cast<size_t>(t) * d4 + c));
                }
            }
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < T * d / 8; i += kDecThreads) {
            const uint4 v = reinterpret_cast<const uint4 *>(xs)[i];
            reinterpret_cast<uint4 *>(a.x_cur)[i] = v;
            if (a.x_export) reinterpret_cast<uint4 *>(a.x_export)[i] = v;
        }
    }
    {
        // fp16 copy in the permuted B layout of the expert GEMVs (8 token columns),
        // split over the CTAs: the 8 elements of one 32-bit weight word land as
        // 16 contiguous bytes (x0 x2 x4 x6 | x1 x3 x5 x7)
        const int wpt = d / 8;  // words per token
        const int per = (8 * wpt + gridDim.x - 1) / gridDim.x;
        for (int q = blockIdx.x * per + threadIdx.x; q < min(8 * wpt, (blockIdx.x + 1) * per); q += kDecThreads) {
            const int n = q / wpt, k0 = (q - n * wpt) * 8;
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (n < T) {
                const uint4 v = *reinterpret_cast<const uint4 *>(xs + static_cast<size_t>(n) * d + k0);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 p2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
                    f[2 * j] = p2.x;
                    f[2 * j + 1] = p2.y;
                }
                const __half2 h0 = __floats2half2_rn(f[0], f[2]), h1 = __floats2half2_rn(f[4], f[6]);
                const __half2 h2 = __floats2half2_rn(f[1], f[3]), h3 = __floats2half2_rn(f[5], f[7]);
                o = make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                               *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
                if (f16x2_has_inf(o.x) | f16x2_has_inf(o.y) | f16x2_has_inf(o.z) | f16x2_has_inf(o.w))
                    record_error(&a.ctrl->status, kErrDeviceRange);
            }
            *reinterpret_cast<uint4 *>(a.xp + perm_b_index(k0, n)) = o;
        }
    }

    // ---- router GEMV: one warp per expert
    if (e < a.E) {
        // compact code (one token per loop trip): this kernel runs once per layer,
        // so its instructions are fetched cold and unrolled copies cost fetch time
        const float bias = a.router_bias ? a.router_bias[e] : 0.0f;
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            const uint4 *xrow = reinterpret_cast<const uint4 *>(xs + static_cast<size_t>(t) * d);
            float acc = 0.0f;
#pragma unroll
            for (int m = 0; m < kPre; ++m) {
                const int c = lane + 32 * m;
                if (c < n8) acc = dot8_bf16(wpre[m], xrow[c], acc);
            }
#pragma unroll 1
            for (int c = lane + 32 * kPre; c < n8; c += 32) acc = dot8_bf16(__ldg(wrow + c), xrow[c], acc);
            const float sum = warp_sum(acc) + bias;
            if (lane == 0) {
                a.logits[t * a.E + e] = sum;
                if (a.trace_logits) a.trace_logits[t * a.E + e] = sum;
            }
        }
    }
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 128-wide K block of a 16-row tile: q_g / q_g8 hold this lane's 16 bytes of
// rows g and g + 8, sb_g / sb_g8 the bf16 scale (low half) and bias (high
// half) of its group; b points at the lane's B fragments of the block
// (8 slices x 4 fp16, consecutive).
__device__ __forceinline__ void mma_kblock(float (&d)[4], uint4 q_g, uint4 q_g8, uint32_t sb_g, uint32_t sb_g8,
                                           const uint2 *b)
{
    const __half2 k8 = __floats2half2_rn(8.0f, 8.0f);
    const __half2 s8_g = __hmul2(half2_from_bf16_bits(static_cast<uint16_t>(sb_g & 0xFFFFu)), k8);
    const __half2 b_g = half2_from_bf16_bits(static_cast<uint16_t>(sb_g >> 16));
    const __half2 s8_g8 = __hmul2(half2_from_bf16_bits(static_cast<uint16_t>(sb_g8 & 0xFFFFu)), k8);
    const __half2 b_g8 = half2_from_bf16_bits(static_cast<uint16_t>(sb_g8 >> 16));
    const uint32_t wg[4] = {q_g.x, q_g.y, q_g.z, q_g.w}, wg8[4] = {q_g8.x, q_g8.y, q_g8.z, q_g8.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint4 pg = dequant8_f16_e2m3(wg[w], s8_g, b_g);
        const uint4 pg8 = dequant8_f16_e2m3(wg8[w], s8_g8, b_g8);
        const uint2 b0 = b[2 * w], b1 = b[2 * w + 1];
        const uint32_t a0[4] = {pg.x, pg8.x, pg.y, pg8.y};  // slice 2w: pairs (0,2) and (4,6)
        const uint32_t a1[4] = {pg.z, pg8.z, pg.w, pg8.w};  // slice 2w + 1: pairs (1,3) and (5,7)
        mma_16816(d, a0, b0.x, b0.y);
        mma_16816(d, a1, b1.x, b1.y);
    }
}

// gate/up: task = (unit, 32 rows of I); warp w takes rows 16 (w % 2) .. + 16
// and the K blocks kb = w / 2 (mod 4), both matrices; the four K-split partial
// tiles are summed in shared memory, then h' = f16(w_u[t] * silu(gate) * up) is
// written in the permuted B layout of the down projection (K = units x I).
__global__ void __launch_bounds__(kDecThreads)
dec_gateup_kernel(const DecodeLayerArgs a)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __half *xp = reinterpret_cast<__half *>(dsm);                                 // [d/128][8][4][8][4]
    float *red = reinterpret_cast<float *>(dsm + static_cast<size_t>(a.d) * 8 * 2);  // [8 warps][2][32][4]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int T = a.T, d = a.d, I = a.I, nkb = d / kKB, ngroups = d / 64;
    const int tpu = I / 32;  // tasks per unit (32 rows of I each)
    const int rt = warp & 1, ks = warp >> 1;

    // One round of weight loads of a task: up to 4 K blocks of this warp, both
    // matrices, rows g and g + 8 of its 16-row tile.  The round's scales and
    // biases (32 groups = 64 bytes of each row) are read as 8-byte pieces of 4
    // groups, pieces t and t + 4 by lane t of the row's quad (coalesced within
    // the quad), and handed to the lane that needs each group by a shuffle.
    uint4 qg[4], qg8[4], qu[4], qu8[4];
    uint2 sbp[8][2];  // [gate g s, b; gate g+8 s, b; up g s, b; up g+8 s, b][piece t, t + 4]
    auto issue_loads = [&](int e, int i0, int kb0) {
        const bool sh = e < 0;
        const size_t row_g = (sh ? 0 : static_cast<size_t>(e) * I) + i0 + g, row_g8 = row_g + 8;
        const uint8_t *gq = sh ? a.sh_gate_q : a.gate_q, *uq = sh ? a.sh_up_q : a.up_q;
        const uint16_t *gs = sh ? a.sh_gate_s : a.gate_s, *gb = sh ? a.sh_gate_b : a.gate_b;
        const uint16_t *us = sh ? a.sh_up_s : a.up_s, *ub = sh ? a.sh_up_b : a.up_b;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int kb = kb0 + 4 * m;
            if (kb < nkb) {
                const size_t off = static_cast<size_t>(kb) * (kKB / 2) + t * 16;
                qg[m] = ld_early(gq + row_g * (d / 2) + off);
                qg8[m] = ld_early(gq + row_g8 * (d / 2) + off);
                qu[m] = ld_early(uq + row_g * (d / 2) + off);
                qu8[m] = ld_early(uq + row_g8 * (d / 2) + off);
            }
        }
        const uint16_t *rows[8] = {gs + row_g * ngroups, gb + row_g * ngroups, gs + row_g8 * ngroups,
                                   gb + row_g8 * ngroups, us + row_g * ngroups, ub + row_g * ngroups,
                                   us + row_g8 * ngroups, ub + row_g8 * ngroups};
        const int p0 = 2 * (kb0 - ks);  // the round's first group
#pragma unroll
        for (int k = 0; k < 8; ++k) {
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const int gp = p0 + 4 * (t + 4 * sl);  // ngroups is a multiple of 4: pieces are whole
                sbp[k][sl] = gp < ngroups ? ld_early8(rows[k] + gp) : make_uint2(0u, 0u);
            }
        }
    };
    // scale (low half) and bias (high half) of group 2 kb + (t >> 1) of row k / 2
    // of sbp, kb = kb0 + 4 m: piece 2 m + ks / 2 of the round, word ks % 2 of it
    auto pick_sb = [&](int k, int m) {
        const int piece = 2 * m + (ks >> 1), src = (lane & ~3) | (piece & 3);
        const uint2 ps = (piece >> 2) ? sbp[k][1] : sbp[k][0], pb = (piece >> 2) ? sbp[k + 1][1] : sbp[k + 1][0];
        const uint32_t ws = __shfl_sync(0xffffffffu, (ks & 1) ? ps.y : ps.x, src);
        const uint32_t wb = __shfl_sync(0xffffffffu, (ks & 1) ? pb.y : pb.x, src);
        const int hi = (t >> 1) & 1;
        return (hi ? ws >> 16 : ws & 0xFFFFu) | ((hi ? wb >> 16 : wb & 0xFFFFu) << 16);
    };
    pdl_trigger();
    // The shared expert is unit 0 and does not depend on the routing: its CTAs
    // issue their first weight loads before waiting for the router.
    const bool preloaded = blockIdx.x < tpu;
    if (preloaded) issue_loads(-1, blockIdx.x * 32 + rt * 16, ks);
    pdl_wait();
    // this token's logits first (the top-8 waits for them), then the fp16 input
    // to shared memory asynchronously; the first round of weight loads is
    // issued before waiting for it
    float4 l0 = make_float4(0.f, 0.f, 0.f, 0.f), l1 = l0;
    if (warp < T) {
        const float4 *src = reinterpret_cast<const float4 *>(a.logits + warp * a.E + lane * 8);
        l0 = __ldcg(src);
        l1 = __ldcg(src + 1);
    }
    for (int i = threadIdx.x; i < d; i += kDecThreads)  // 8 x d fp16 = d uint4
        cp_async_16(reinterpret_cast<uint4 *>(xp) + i, reinterpret_cast<const uint4 *>(a.xp) + i);
    cp_async_commit();
    bool xp_ready = false;

    // Top-8 per token and the list of distinct experts ("units": the shared
    // expert first with weight 1, then the routed experts ascending), computed by
    // every CTA from the logits;
    // CTA 0 publishes it for the down projection and the trace.
    __shared__ int umask[256];
    __shared__ float uw[256][kMaxT];
    __shared__ int scan_tmp[kDecWarps];
    __shared__ int s_expert[kMaxT * 8 + 1];
    __shared__ float s_w[kMaxT * 8 + 1][kMaxT];
    __shared__ int s_n_units;
    umask[threadIdx.x] = 0;
#pragma unroll
    for (int q = 0; q < kMaxT; ++q) uw[threadIdx.x][q] = 0.0f;
    __syncthreads();
    if (warp < T) {
        const int tok = warp;
        const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
        int sel_e;
        float sel_w;
        warp_top8_keys(lv, lane, sel_e, sel_w);
        if (lane < 8) {
            if (blockIdx.x == 0 && a.trace_idx) a.trace_idx[tok * 8 + lane] = sel_e;
            if (blockIdx.x == 0 && a.trace_w) a.trace_w[tok * 8 + lane] = sel_w;
            atomicOr(&umask[sel_e], 1 << tok);
            uw[sel_e][tok] = sel_w;
        }
    }
    __syncthreads();
    {
        const int used = umask[threadIdx.x] != 0;
        int incl = used;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nb = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += nb;
        }
        if (lane == 31) scan_tmp[warp] = incl;
        __syncthreads();
        int off = 0, n_used = 0;
        for (int w = 0; w < kDecWarps; ++w) {
            if (w < warp) off += scan_tmp[w];
            n_used += scan_tmp[w];
        }
        const int u = 1 + off + incl - used;
        if (used) {
            s_expert[u] = threadIdx.x;
#pragma unroll
            for (int q = 0; q < kMaxT; ++q) s_w[u][q] = uw[threadIdx.x][q];
            if (blockIdx.x == 0) {
                a.unit_expert[u] = threadIdx.x;
                a.unit_mask[u] = umask[threadIdx.x];
#pragma unroll
                for (int q = 0; q < kMaxT; ++q) a.unit_w[u * kMaxT + q] = uw[threadIdx.x][q];
            }
        }
        if (threadIdx.x == 0) {
            s_expert[0] = -1;  // shared expert
#pragma unroll
            for (int q = 0; q < kMaxT; ++q) s_w[0][q] = 1.0f;
            s_n_units = n_used + 1;
            if (blockIdx.x == 0) {
                a.unit_expert[0] = -1;
                a.unit_mask[0] = (1 << T) - 1;
#pragma unroll
                for (int q = 0; q < kMaxT; ++q) a.unit_w[q] = 1.0f;
                *a.n_units = n_used + 1;
            }
        }
        __syncthreads();
    }
    const int n_units = s_n_units;
    if (blockIdx.x >= n_units * tpu) {
        cp_async_wait_all();  // no copy into shared memory in flight at exit
        return;
    }
    for (int task = blockIdx.x; task < n_units * tpu; task += gridDim.x) {
        const int u = task / tpu;
        const int i0 = (task - u * tpu) * 32 + rt * 16;
        const int e = s_expert[u];
        float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r0 = 0; r0 < nkb; r0 += 4 * 4) {  // rounds: the same count in every warp
            const int kb0 = r0 + ks;
            // up to 4 K blocks of this warp: all loads first, then the MMAs
            if (!(preloaded && task == blockIdx.x && r0 == 0)) issue_loads(e, i0, kb0);
            if (!xp_ready) {
                cp_async_wait_all();
                __syncthreads();
                xp_ready = true;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int kb = kb0 + 4 * m;
                if (kb < nkb) {
                    const uint2 *bf = reinterpret_cast<const uint2 *>(xp + (((kb * 8 + g) * 4 + t) * 8) * 4);
                    mma_kblock(accg, qg[m], qg8[m], pick_sb(0, m), pick_sb(2, m), bf);
                    mma_kblock(accu, qu[m], qu8[m], pick_sb(4, m), pick_sb(6, m), bf);
                }
            }
        }
        // sum the four K-split partial tiles of each row tile
        float *mine = red + (warp * 2) * 32 * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mine[lane * 4 + q] = accg[q];
            mine[32 * 4 + lane * 4 + q] = accu[q];
        }
        __syncthreads();
        if (ks == 0) {
#pragma unroll
            for (int p = 1; p < 4; ++p) {
                const float *o = red + ((rt + 2 * p) * 2) * 32 * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    accg[q] += o[lane * 4 + q];
                    accu[q] += o[32 * 4 + lane * 4 + q];
                }
            }
            // fragment: q = 0/1 -> row g, tokens 2t, 2t+1; q = 2/3 -> row g + 8
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = 2 * t + (q & 1);
                const int i = i0 + g + 8 * (q >> 1);
                const float wt = s_w[u][n];
                const float hv = wt * silu_f(accg[q]) * accu[q];
                const __half hh = __float2half_rn(hv);
                if (__hisinf(hh)) record_error(&a.ctrl->status, kErrDeviceRange);
                a.h[perm_b_index(u * I + i, n)] = hh;
            }
        }
        __syncthreads();
    }
}

// down: task = 16 output rows; the 8 warps split the K blocks of
// K = units x I (unit u, block j), accumulate in one tile, and the partial
// tiles are summed in shared memory.  out[t][row] = sum over units of
// Wd_u[row] . h'_u[t] (the routing weight is already in h').
constexpr int kDownWarps = 16;  // 512 threads: every K block of a row tile in flight at once for T = 1

__global__ void __launch_bounds__(kDownWarps * 32)
dec_down_kernel(const DecodeLayerArgs a)
{
    __shared__ float red[kDownWarps][32][4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int T = a.T, d = a.d, I = a.I, kpu = I / kKB, ngroups = I / 64;
    uint4 q[3], q8[3];
    // scale / bias of K block jb: groups 2 jb and 2 jb + 1 (one 32-bit word) of
    // rows j0 + g and j0 + g + 8; lane t of a row's quad loads word t of
    // {scale row, bias row, scale row + 8, bias row + 8}, shuffles share them
    uint32_t sbw[3];
    uint2 bfr[3][8];
    // weight loads of K block kb (unit u, block jb) for output rows j0 + g, j0 + g + 8
    auto load_w = [&](int m, int e, int jb, int j0) {
        const bool sh = e < 0;
        const size_t row = (sh ? 0 : static_cast<size_t>(e) * d) + j0 + g;
        const uint8_t *dq = sh ? a.sh_down_q : a.down_q;
        const uint16_t *ds = sh ? a.sh_down_s : a.down_s, *db = sh ? a.sh_down_b : a.down_b;
        const size_t off = static_cast<size_t>(jb) * (kKB / 2) + t * 16;
        q[m] = ld_early(dq + row * (I / 2) + off);
        q8[m] = ld_early(dq + (row + 8) * (I / 2) + off);
        const uint16_t *w = (t & 1 ? db : ds) + (row + 8 * (t >> 1)) * ngroups + 2 * jb;
        sbw[m] = ld_early_u32(w);
    };
    pdl_trigger();
    // unit 0 is the shared expert: the warps whose first K block lies in it issue
    // those weight loads before waiting for the gate/up kernel
    const bool preloaded = warp < kpu && blockIdx.x < d / 16;
    if (preloaded) load_w(0, -1, warp, blockIdx.x * 16);
    pdl_wait();
    const int n_units = *a.n_units;
    if (n_units < 1 || n_units > a.top_k * T + 1) {  // the h buffer holds top_k * T + 1 units
        if (threadIdx.x == 0) record_error(&a.ctrl->status, kErrDeviceIndex);
        return;
    }
    const int n_kb = n_units * kpu;
    for (int task = blockIdx.x; task < d / 16; task += gridDim.x) {
        const int j0 = task * 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kb0 = warp; kb0 < n_kb; kb0 += 3 * kDownWarps) {
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const int kb = kb0 + m * kDownWarps;
                if (kb < n_kb) {
                    const int u = kb / kpu, jb = kb - u * kpu;
                    if (!(preloaded && m == 0 && task == blockIdx.x && kb0 == warp)) {
                        int e = a.unit_expert[u];
                        if (e >= a.E) {
                            if (lane == 0) record_error(&a.ctrl->status, kErrDeviceIndex);
                            e = 0;
                        }
                        load_w(m, e, jb, j0);
                    }
                    // token column g of h' is zero for g >= T: no load.  The lane's 8
                    // fragments are 64 contiguous bytes: four 16-byte loads
                    const uint4 *src = reinterpret_cast<const uint4 *>(a.h) + ((kb * 8 + g) * 4 + t) * 4;
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        const uint4 v = g < T ? __ldcg(src + s2) : make_uint4(0u, 0u, 0u, 0u);
                        bfr[m][2 * s2] = make_uint2(v.x, v.y);
                        bfr[m][2 * s2 + 1] = make_uint2(v.z, v.w);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                if (kb0 + m * kDownWarps < n_kb) {
                    const int quad = lane & ~3, hi = (t >> 1) & 1;
                    uint32_t wv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t v = __shfl_sync(0xffffffffu, sbw[m], quad + k);
                        wv[k] = hi ? v >> 16 : v & 0xFFFFu;
                    }
                    mma_kblock(acc, q[m], q8[m], wv[0] | (wv[1] << 16), wv[2] | (wv[3] << 16), bfr[m]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) red[warp][lane][q] = acc[q];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int p = 1; p < kDownWarps; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[q] += red[p][lane][q];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = 2 * t + (q & 1);
                if (n < T) a.out[static_cast<size_t>(n) * d + j0 + g + 8 * (q >> 1)] = acc[q];
            }
        }
        __syncthreads();
    }
}

// Dynamic shared memory: the router kernel stages the bf16 inputs [T][d]; the
// gate/up kernel the fp16 inputs of up to 8 tokens in the permuted B layout
// plus the per-warp partial sums [warps][2][32][4] floats.
size_t decode_smem_route(int T, int d) { return static_cast<size_t>(T) * d * 2; }
size_t decode_smem_gateup(int d) { return static_cast<size_t>(d) * 8 * 2 + kDecWarps * 2 * 32 * 4 * 4; }

}  // namespace

cudaError_t launch_decode_layer(const DecodeLayerArgs &a, int num_sms, cudaStream_t stream)
{
    for (const void *k : {reinterpret_cast<const void *>(dec_route_kernel<4>), reinterpret_cast<const void *>(dec_route_kernel<8>),
                          reinterpret_cast<const void *>(dec_gateup_kernel), reinterpret_cast<const void *>(dec_down_kernel)}) {
        const cudaError_t e = set_max_dynamic_smem(k, 200 * 1024);
        if (e != cudaSuccess) return e;
    }
    // programmatic dependent launches: each kernel starts while its predecessor finishes
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kDecThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    cfg.gridDim = dim3((a.E + kDecWarps - 1) / kDecWarps);
    cfg.dynamicSmemBytes = decode_smem_route(a.T, a.d);
    const int J = (a.d / 4 + kDecThreads - 1) / kDecThreads;  // float4 of the previous output per thread and token
    if ((e = cudaLaunchKernelEx(&cfg, a.T * J <= 4 ? dec_route_kernel<4> : dec_route_kernel<8>, a)) != cudaSuccess) return e;
    cfg.gridDim = dim3(num_sms);
    cfg.dynamicSmemBytes = decode_smem_gateup(a.d);
    if ((e = cudaLaunchKernelEx(&cfg, dec_gateup_kernel, a)) != cudaSuccess) return e;
    cfg.gridDim = dim3(std::min(num_sms, a.d / 16));
    cfg.blockDim = dim3(kDownWarps * 32);
    cfg.dynamicSmemBytes = 0;
    if ((e = cudaLaunchKernelEx(&cfg, dec_down_kernel, a)) != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lily

namespace lily {
namespace {

// Final export of the decode chain: x_next = bf16(out / sqrt(mean(out^2) + 1e-6)).
__global__ void __launch_bounds__(256) dec_final_norm_kernel(const float *prev_out, uint16_t *x_export, int d)
{
    __shared__ float red[8];
    const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *row = prev_out + static_cast<size_t>(t) * d;
    float ss = 0.0f;
    for (int c = threadIdx.x; c < d; c += 256) ss = fmaf(row[c], row[c], ss);
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float s = 0.0f;
    for (int w = 0; w < 8; ++w) s += red[w];
    const float inv = 1.0f / sqrtf(s / static_cast<float>(d) + 1e-6f);
    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(x_export) + static_cast<size_t>(t) * d;
    for (int c = threadIdx.x; c < d; c += 256) dst[c] = __float2bfloat16_rn(row[c] * inv);
}

}  // namespace

cudaError_t launch_decode_final_norm(const float *prev_out, uint16_t *x_export, int T, int d, cudaStream_t stream)
{
    dec_final_norm_kernel<<<T, 256, 0, stream>>>(prev_out, x_export, d);
    return cudaGetLastError();
}

}  // namespace lily
