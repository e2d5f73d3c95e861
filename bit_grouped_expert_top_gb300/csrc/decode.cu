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
//                       to bf16), router GEMV (one warp per expert), and in the
//                       last CTA the top-8 selection per token and the list of
//                       distinct experts ("units") with per-token weights; the
//                       shared expert is the last unit with weight 1.
//   dec_gateup_kernel : one warp per (unit, intermediate row): gate and up rows
//                       dequantised and dotted with the unit's tokens, SwiGLU,
//                       h stored as fp16.
//   dec_down_kernel   : one warp per output row: the down rows of every unit,
//                       dotted with h, scaled by the routing weight and summed
//                       in registers (deterministic, no atomics).
#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxT = 8;
constexpr int kChunk = 32;       // weights per 16-byte int4 chunk
constexpr int kPadChunk = 40;    // bf16 elements per chunk slot in shared memory (80 B: bank-conflict-free)

// Shared-memory copy of activations: [rows][n_chunks][kPadChunk] bf16.
__device__ __forceinline__ int pad_index(int row, int k, int n_chunks)
{
    return (row * n_chunks + (k >> 5)) * kPadChunk + (k & 31);
}

// 16-bit activation pair -> float2 (bf16 layer input or fp16 h).
__device__ __forceinline__ float2 act2_to_float2(uint32_t u, const __nv_bfloat16 *)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ float2 act2_to_float2(uint32_t u, const __half *)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}

// dot of 32 dequantised weights (one 16-byte int4 chunk; each weight rounded
// once to fp16, as in the prefill path) with 32 activations stored
// contiguously in shared memory; fp32 accumulation.
template <typename Act>
__device__ __forceinline__ float dot32(const uint4 q, __half2 s2, __half2 b2, const Act *xs)
{
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    const uint4 *xv = reinterpret_cast<const uint4 *>(xs);
    float acc = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 wv = dequant8_f16(words[c], s2, b2);
        const uint4 x8 = xv[c];
        const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t xu[4] = {x8.x, x8.y, x8.z, x8.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&wu[p]));
            const float2 xf = act2_to_float2(xu[p], xs);
            acc = fmaf(wf.x, xf.x, acc);
            acc = fmaf(wf.y, xf.y, acc);
        }
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kDecThreads)
dec_route_kernel(const DecodeLayerArgs a)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(dsm);  // [T][d] plain layout
    __shared__ float red[kDecWarps][kMaxT];
    __shared__ float inv_rms[kMaxT];
    __shared__ int is_last;
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
        if (e < a.E && c < n8) wpre[m] = __ldg(wrow + c);
    }

    // ---- layer input
    if (a.prev_out == nullptr) {
        for (int i = threadIdx.x; i < T * d / 8; i += kDecThreads)
            reinterpret_cast<uint4 *>(xs)[i] = reinterpret_cast<const uint4 *>(a.x_in)[i];
    } else {
        float ss[kMaxT];
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) ss[t] = 0.0f;
#pragma unroll 4
        for (int c = threadIdx.x; c < d; c += kDecThreads) {
#pragma unroll
            for (int t = 0; t < kMaxT; ++t)
                if (t < T) {
                    const float v = a.prev_out[static_cast<size_t>(t) * d + c];
                    ss[t] = fmaf(v, v, ss[t]);
                }
        }
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            const float s = warp_sum(ss[t]);
            if (lane == 0) red[warp][t] = s;
        }
        __syncthreads();
        if (threadIdx.x < T) {
            float s = 0.0f;
            for (int w = 0; w < kDecWarps; ++w) s += red[w][threadIdx.x];
            inv_rms[threadIdx.x] = 1.0f / sqrtf(s / static_cast<float>(d) + 1e-6f);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < T * d; i += kDecThreads) {
            const int t = i / d;
            xs[i] = __float2bfloat16_rn(a.prev_out[i] * inv_rms[t]);
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

    // ---- router GEMV: one warp per expert
    if (e < a.E) {
        float acc[kMaxT];
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) acc[t] = 0.0f;
        for (int m0 = 0; m0 * 32 < n8; m0 += kPre) {
#pragma unroll
            for (int m = 0; m < kPre; ++m) {
                const int c = lane + 32 * (m0 + m);
                if (c >= n8) continue;
                const uint4 wv = m0 == 0 ? wpre[m] : __ldg(wrow + c);
                const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int t = 0; t < kMaxT; ++t) {
                    if (t < T) {
                        const uint4 xv = reinterpret_cast<const uint4 *>(xs + static_cast<size_t>(t) * d)[c];
                        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wu[p]));
                            const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xu[p]));
                            acc[t] = fmaf(wf.x, xf.x, acc[t]);
                            acc[t] = fmaf(wf.y, xf.y, acc[t]);
                        }
                    }
                }
            }
        }
        const float bias = a.router_bias ? a.router_bias[e] : 0.0f;
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
                const float s = warp_sum(acc[t]) + bias;
                if (lane == 0) {
                    a.logits[t * a.E + e] = s;
                    if (a.trace_logits) a.trace_logits[t * a.E + e] = s;
                }
            }
        }
    }

    // ---- last CTA: top-8 per token and the unit list
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(&a.ctrl->ticket2, 1u);
        is_last = (prev == static_cast<unsigned int>(gridDim.x) - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    __shared__ int umask[256];
    __shared__ float uw[256][kMaxT];
    __shared__ int scan_tmp[kDecWarps];
    umask[threadIdx.x] = 0;
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) uw[threadIdx.x][t] = 0.0f;
    __syncthreads();
    if (warp < T) {
        const int t = warp;
        int sel_e;
        float sel_w;
        warp_top8_of_256(a.logits + t * a.E, lane, sel_e, sel_w);
        if (lane < 8) {
            if (a.trace_idx) a.trace_idx[t * 8 + lane] = sel_e;
            if (a.trace_w) a.trace_w[t * 8 + lane] = sel_w;
            atomicOr(&umask[sel_e], 1 << t);
            uw[sel_e][t] = sel_w;
        }
    }
    __syncthreads();
    // compact the used experts in ascending order
    const int used = umask[threadIdx.x] != 0;
    int incl = used;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    int off = 0, n_used = 0;
    for (int w = 0; w < kDecWarps; ++w) {
        if (w < warp) off += scan_tmp[w];
        n_used += scan_tmp[w];
    }
    const int u = off + incl - used;
    if (used) {
        a.unit_expert[u] = threadIdx.x;
        a.unit_mask[u] = umask[threadIdx.x];
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) a.unit_w[u * kMaxT + t] = uw[threadIdx.x][t];
    }
    if (threadIdx.x == 0) {
        a.unit_expert[n_used] = -1;  // shared expert
        a.unit_mask[n_used] = (1 << T) - 1;
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) a.unit_w[n_used * kMaxT + t] = 1.0f;
        *a.n_units = n_used + 1;
        a.ctrl->ticket2 = 0u;
    }
}

// Loads the layer input x_cur [T][d] into the padded shared layout.
template <typename Act>
__device__ __forceinline__ void load_padded(const uint16_t *src, Act *dst, int rows, int K)
{
    const int n_chunks = K / kChunk;
    for (int i = threadIdx.x; i < rows * K / 8; i += kDecThreads) {
        const int row = (i * 8) / K, k = (i * 8) % K;
        *reinterpret_cast<uint4 *>(dst + pad_index(row, k, n_chunks)) = reinterpret_cast<const uint4 *>(src)[i];
    }
}

__global__ void __launch_bounds__(kDecThreads, 2)
dec_gateup_kernel(const DecodeLayerArgs a)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(dsm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = a.T, d = a.d, I = a.I;
    const int n_chunks = d / kChunk, ngroups = d / 64;
    load_padded(a.x_cur, xs, T, d);
    __syncthreads();

    const int n_units = *a.n_units;
    const int items = n_units * I;
    const int n_pairs = (items + 1) / 2;
    // A warp takes two (unit, row) items at a time; each lane first issues every
    // 16-byte weight load of both items (gate and up), then computes.
    for (int pr = blockIdx.x * kDecWarps + warp; pr < n_pairs; pr += gridDim.x * kDecWarps) {
        const uint4 *gq[2], *uq[2];
        const uint16_t *gs[2], *gb[2], *us[2], *ub[2];
        int mask[2], uu[2], ii[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int item = min(2 * pr + k, items - 1);
            const int u = item / I, i = item - u * I;
            const int e = a.unit_expert[u];
            int m = a.unit_mask[u] & ((1 << T) - 1);
            if (e >= a.E || m == 0) {
                if (lane == 0) record_error(&a.ctrl->status, kErrDeviceIndex);
                m = 0;
            }
            if (2 * pr + k >= items) m = 0;  // odd tail: the duplicate item does nothing
            const bool sh = e < 0;
            const size_t row = sh ? static_cast<size_t>(i) : static_cast<size_t>(e < a.E ? e : 0) * I + i;
            gq[k] = reinterpret_cast<const uint4 *>((sh ? a.sh_gate_q : a.gate_q) + row * (d / 2));
            uq[k] = reinterpret_cast<const uint4 *>((sh ? a.sh_up_q : a.up_q) + row * (d / 2));
            gs[k] = (sh ? a.sh_gate_s : a.gate_s) + row * ngroups;
            gb[k] = (sh ? a.sh_gate_b : a.gate_b) + row * ngroups;
            us[k] = (sh ? a.sh_up_s : a.up_s) + row * ngroups;
            ub[k] = (sh ? a.sh_up_b : a.up_b) + row * ngroups;
            mask[k] = m;
            uu[k] = u;
            ii[k] = i;
        }
        float accg[2][kMaxT], accu[2][kMaxT];
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int t = 0; t < kMaxT; ++t) accg[k][t] = accu[k][t] = 0.0f;
        for (int c0 = 0; c0 < n_chunks; c0 += 2 * 32) {
            uint4 qg[2][2], qu[2][2];
            uint16_t vgs[2][2], vgb[2][2], vus[2][2], vub[2][2];
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int c = c0 + q * 32 + lane;
                    if (c < n_chunks && mask[k]) {
                        qg[k][q] = __ldg(gq[k] + c);
                        qu[k][q] = __ldg(uq[k] + c);
                        vgs[k][q] = __ldg(gs[k] + (c >> 1));
                        vgb[k][q] = __ldg(gb[k] + (c >> 1));
                        vus[k][q] = __ldg(us[k] + (c >> 1));
                        vub[k][q] = __ldg(ub[k] + (c >> 1));
                    }
                }
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int c = c0 + q * 32 + lane;
                    if (c < n_chunks && mask[k]) {
                        const __half2 sg = half2_from_bf16_bits(vgs[k][q]), bg = half2_from_bf16_bits(vgb[k][q]);
                        const __half2 su = half2_from_bf16_bits(vus[k][q]), bu = half2_from_bf16_bits(vub[k][q]);
#pragma unroll
                        for (int t = 0; t < kMaxT; ++t) {
                            if (t < T && ((mask[k] >> t) & 1)) {
                                const __nv_bfloat16 *xr = xs + pad_index(t, c * kChunk, n_chunks);
                                accg[k][t] += dot32(qg[k][q], sg, bg, xr);
                                accu[k][t] += dot32(qu[k][q], su, bu, xr);
                            }
                        }
                    }
                }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int t = 0; t < kMaxT; ++t) {
                if (t < T && ((mask[k] >> t) & 1)) {
                    const float gv = warp_sum(accg[k][t]);
                    const float uv = warp_sum(accu[k][t]);
                    if (lane == 0)
                        a.h[(static_cast<size_t>(uu[k]) * kMaxT + t) * I + ii[k]] = __float2half_rn(silu_f(gv) * uv);
                }
            }
    }
}

__global__ void __launch_bounds__(kDecThreads)
dec_down_kernel(const DecodeLayerArgs a)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __half *hs = reinterpret_cast<__half *>(dsm);  // compact (unit, token) rows of h, padded
    __shared__ int s_expert[kMaxT * 8 + 1];
    __shared__ int s_mask[kMaxT * 8 + 1];
    __shared__ int s_slot[kMaxT * 8 + 1];  // first compact h slot of each unit
    __shared__ float s_w[kMaxT * 8 + 1][kMaxT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = a.T, d = a.d, I = a.I;
    const int n_chunks = I / kChunk, ngroups = I / 64;
    const int n_units = *a.n_units;
    if (n_units < 1 || n_units > kMaxT * 8 + 1) {
        if (threadIdx.x == 0) record_error(&a.ctrl->status, kErrDeviceIndex);
        return;
    }
    for (int u = threadIdx.x; u < n_units; u += kDecThreads) {
        s_expert[u] = a.unit_expert[u];
        s_mask[u] = a.unit_mask[u] & ((1 << T) - 1);
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) s_w[u][t] = a.unit_w[u * kMaxT + t];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int u = 0; u < n_units; ++u) {
            s_slot[u] = run;
            run += __popc(s_mask[u]);
        }
    }
    __syncthreads();
    // Compact copy of h: one padded row per (unit, token served by the unit).
    for (int u = warp; u < n_units; u += kDecWarps) {
        const int mask = s_mask[u];
        int slot = s_slot[u];
        for (int t = 0; t < T; ++t) {
            if (!((mask >> t) & 1)) continue;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.h + (static_cast<size_t>(u) * kMaxT + t) * I);
            for (int i = lane; i < I / 8; i += 32)
                *reinterpret_cast<uint4 *>(hs + pad_index(slot, i * 8, n_chunks)) = src[i];
            ++slot;
        }
    }
    __syncthreads();

    for (int j = blockIdx.x * kDecWarps + warp; j < d; j += gridDim.x * kDecWarps) {
        float acc[kMaxT];
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) acc[t] = 0.0f;
        const int n_items = n_units * n_chunks;
        constexpr int kB = 8;  // chunk-items per lane with loads in flight together
        for (int it0 = 0; it0 < n_items; it0 += kB * 32) {
            uint4 q[kB];
            uint16_t vs[kB], vb[kB];
#pragma unroll
            for (int m = 0; m < kB; ++m) {
                const int it = it0 + m * 32 + lane;
                if (it < n_items) {
                    const int u = it / n_chunks, c = it - u * n_chunks;
                    const int e = s_expert[u];
                    const bool sh = e < 0;
                    const size_t row = sh ? static_cast<size_t>(j) : static_cast<size_t>(e) * d + j;
                    q[m] = __ldg(reinterpret_cast<const uint4 *>((sh ? a.sh_down_q : a.down_q) + row * (I / 2)) + c);
                    vs[m] = __ldg((sh ? a.sh_down_s : a.down_s) + row * ngroups + (c >> 1));
                    vb[m] = __ldg((sh ? a.sh_down_b : a.down_b) + row * ngroups + (c >> 1));
                }
            }
#pragma unroll
            for (int m = 0; m < kB; ++m) {
                const int it = it0 + m * 32 + lane;
                if (it < n_items) {
                    const int u = it / n_chunks, c = it - u * n_chunks;
                    const __half2 s2 = half2_from_bf16_bits(vs[m]), b2 = half2_from_bf16_bits(vb[m]);
                    const int mask = s_mask[u];
                    int slot = s_slot[u];
#pragma unroll
                    for (int t = 0; t < kMaxT; ++t) {
                        if (t < T && ((mask >> t) & 1)) {
                            acc[t] += s_w[u][t] * dot32(q[m], s2, b2, hs + pad_index(slot, c * kChunk, n_chunks));
                            ++slot;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
                const float sm = warp_sum(acc[t]);
                if (lane == 0) a.out[static_cast<size_t>(t) * d + j] = sm;
            }
        }
    }
}

}  // namespace

size_t decode_smem_route(int T, int d) { return static_cast<size_t>(T) * d * 2; }
size_t decode_smem_gateup(int T, int d) { return static_cast<size_t>(T) * (d / kChunk) * kPadChunk * 2; }
size_t decode_smem_down(int T, int I) { return static_cast<size_t>(T * 8 + T) * (I / kChunk) * kPadChunk * 2; }

cudaError_t launch_decode_layer(const DecodeLayerArgs &a, int num_sms, cudaStream_t stream)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e;
        if ((e = cudaFuncSetAttribute(dec_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(dec_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(dec_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) != cudaSuccess) return e;
        configured = true;
    }
    dec_route_kernel<<<(a.E + kDecWarps - 1) / kDecWarps, kDecThreads, decode_smem_route(a.T, a.d), stream>>>(a);
    dec_gateup_kernel<<<2 * num_sms, kDecThreads, decode_smem_gateup(a.T, a.d), stream>>>(a);
    dec_down_kernel<<<(a.d + kDecWarps - 1) / kDecWarps, kDecThreads, decode_smem_down(a.T, a.I), stream>>>(a);
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
