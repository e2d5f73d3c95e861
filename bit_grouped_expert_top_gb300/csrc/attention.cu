// Grouped-query decode attention over a fixed-block KV cache, for sm_103a.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br): the model's
// full-attention layers use grouped-query attention, 16 query heads over two
// KV heads, over a growing KV cache (section "O modelo em tres formatos de
// carga"); at decode the page packs the query heads of a KV head together
// (GQA packing), reads the cache coalesced and keeps it in fixed-size blocks
// (section "Prefill e decode: onde estao os ganhos").  Per query head h of a
// sequence:  o_h = sum_t softmax_t(scale q_h . k_{g,t}) v_{g,t},
// g = h / (H_q / H_kv).
//
// GB300 design.  Decode attention is a stream over the cache: each K and V
// byte is read once and used by the (up to 8) query heads of its KV head, so
// HBM bandwidth is the bound.  Split-K over the cache blocks (flash decoding):
// CTA (split, KV head, sequence) owns a contiguous run of the sequence's
// blocks, and a second kernel merges the splits, so a single sequence fills
// the GPU.  Inside a CTA:
//   warp 4      producer: per cache block, TMA copies of its K and V tiles
//               (each [block_size rows][D], as D/64 boxes of 128-byte rows with
//               the 128-byte swizzle) into a ring of shared-memory stages;
//   warps 0..3  consumers, per block:
//               S^T = K q^T on mma.sync m16n8k16 (bf16 in, fp32 out): the
//               block's tokens on the M side (16 per tile, one tile per warp
//               and pass), the 8 query heads of the group on the N side
//               (GQA packing: one K read serves all of them), D on K;
//               online softmax per head in base 2 (running max m, running sum
//               l, the block's max and sum exchanged through shared memory);
//               the weights P, rounded to bf16 (the sum l adds the rounded
//               values, so the weights stay normalised), to shared memory
//               [head][token];
//               O^T += V^T P: D on the M side (each warp a quarter of D), the
//               heads on N, the block's tokens on K; V^T fragments come from
//               ldmatrix.trans on the V tile.
// The partial (m, l, O) of each split goes to the workspace; the combine
// kernel rescales the splits to a common max and normalises.
// Every mbarrier wait is bounded; a wait that gives up records
// LILY_ERR_DEVICE_TIMEOUT and the CTA stops consuming (the producer still
// waits for the copies it issued before it exits).
#include <algorithm>
#include <cmath>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kAttnCW = 4;                          // consumer warps
constexpr int kAttnThreads = (kAttnCW + 1) * 32;    // + the producer warp
constexpr int kAttnMaxStages = 4;
constexpr int kAttnRingBytes = 200 * 1024;          // shared memory for the K/V ring
constexpr int kBarConsumers = 1;                    // named barrier of the consumer warps

// Shared memory besides the ring.
struct AttnSmem {
    uint64_t full[kAttnMaxStages], empty[kAttnMaxStages];
    int abort;
    float red_max[kAttnCW][kAttnMaxGroup];
    float red_sum[kAttnCW][kAttnMaxGroup];
    uint16_t P[kAttnMaxGroup][128 + 8];  // weights of the current block, bf16 [head][token] (rows padded)
};
constexpr size_t kAttnFixed = (sizeof(AttnSmem) + 1023) / 1024 * 1024;

__host__ __device__ inline int stage_bytes(int D, int bs) { return 2 * bs * D * 2; }  // K and V tiles

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += a b: m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset, inside a tile of D/64 swizzled boxes ([bs rows][128 bytes] each),
// of the 16-byte chunk holding elements d .. d + 7 of row r.
__device__ __forceinline__ uint32_t tile_off(int r, int d, int bs)
{
    const int box = d >> 6, c = (d & 63) >> 3;
    return static_cast<uint32_t>(box * bs * 128 + r * 128 + ((c ^ (r & 7)) << 4));
}


__host__ __device__ inline int stages_for(int D, int bs)
{
    if ((D != 64 && D != 128 && D != 256) || (bs != 32 && bs != 64 && bs != 128)) return 0;
    const int fit = kAttnRingBytes / stage_bytes(D, bs);
    const int n = fit < kAttnMaxStages ? fit : kAttnMaxStages;
    return n >= 2 ? n : 0;
}

// Bounded wait on the exit path (ignores the abort flag).
__device__ __forceinline__ void attn_drain_wait(uint64_t *bar, uint32_t parity, int *status)
{
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(addr, parity)) {
        if (global_timer_ns() - t0 > LILY_DRAIN_LIMIT_NS) {
            record_error(status, kErrDeviceTimeout);
            return;
        }
    }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
attn_split_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV)
{
    extern __shared__ uint8_t dsm_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    AttnSmem &S = *reinterpret_cast<AttnSmem *>(base);
    uint8_t *ring = base + kAttnFixed;
    const int D = a.D, bs = a.bs, G = a.group;
    const int NS = stages_for(D, bs), SB = stage_bytes(D, bs);
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
    int *status = &a.ctrl->status;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kAttnCW);
        }
        S.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();  // q, the tables and the cache may come from the previous kernel

    int L = a.seq_lens[b];
    const int cap = a.max_blocks * bs;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0) record_error(status, kErrDeviceIndex);
        L = L < 0 ? 0 : cap;
    }
    const int nblk = (L + bs - 1) / bs;
    const int j0 = static_cast<int>(static_cast<long long>(s) * nblk / a.n_splits);
    const int j1 = static_cast<int>(static_cast<long long>(s + 1) * nblk / a.n_splits);
    const int nb = j1 - j0;
    const size_t pidx = (static_cast<size_t>(b) * a.H_kv + g) * a.n_splits + s;

    if (warp == kAttnCW) {
        // ------------------------------------------------ producer (one thread)
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int issued = 0;
            for (int i = 0; i < nb; ++i) {
                const int slot = i % NS;
                if (i >= NS && !mbar_wait(&S.empty[slot], ((i / NS) - 1) & 1, &S.abort, status)) break;
                int pb = a.block_table[static_cast<size_t>(b) * a.max_blocks + j0 + i];
                if (pb < 0 || pb >= a.n_cache_blocks) {
                    record_error(status, kErrDeviceIndex);
                    pb = 0;
                }
                const int row = (pb * a.H_kv + g) * bs;
                mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(SB));
                uint8_t *kt = ring + static_cast<size_t>(slot) * SB, *vt = kt + SB / 2;
                for (int x = 0; x < D / 64; ++x) {
                    tma_load_2d(kt + x * bs * 128, &tmK, &S.full[slot], x * 64, row);
                    tma_load_2d(vt + x * bs * 128, &tmV, &S.full[slot], x * 64, row);
                }
                ++issued;
            }
            // no copy into this CTA's shared memory may still be in flight at exit
            for (int i = issued > NS ? issued - NS : 0; i < issued; ++i) attn_drain_wait(&S.full[i % NS], (i / NS) & 1, status);
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------- consumers (4 warps)
    // q fragments, the B operand of S^T = K q^T: column n = head gi of the group
    // (zero past the group), rows k = d: d = 16 kk + 2t, +1 and 16 kk + 2t + 8, +9
    const int nks = D / 16, n_mt = bs / 16, mpw = D / 16 / kAttnCW;
    uint32_t qb[16][2];
    {
        const uint16_t *qh = a.q + (static_cast<size_t>(b) * a.H_q + g * G + (gi < G ? gi : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            qb[kk][0] = qb[kk][1] = 0u;
            if (kk < nks && gi < G) {
                qb[kk][0] = *reinterpret_cast<const uint32_t *>(qh + kk * 16 + 2 * t);
                qb[kk][1] = *reinterpret_cast<const uint32_t *>(qh + kk * 16 + 2 * t + 8);
            }
        }
    }
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.0f, l_run1 = 0.0f;  // heads 2t, 2t + 1
    float acc[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[x][c] = 0.0f;
    bool ok = true;

    for (int i = 0; i < nb; ++i) {
        const int slot = i % NS;
        int got = 0;
        if (lane == 0) got = ok && mbar_wait(&S.full[slot], (i / NS) & 1, &S.abort, status);
        ok = __shfl_sync(0xffffffffu, got, 0) != 0;
        const uint32_t kt_s = smem_u32(ring + static_cast<size_t>(slot) * SB), vt_s = kt_s + SB / 2;
        const int tok_base = (j0 + i) * bs;

        // ---- scores of this warp's token tiles (base-2 logits), masked past L
        float sc[2][4];
        float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int mt = warp + kAttnCW * mi;
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[mi][c] = -INFINITY;
            if (ok && mt < n_mt) {
                float c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    if (kk < nks) {
                        uint32_t af[4];
                        ldmatrix_x4(af, kt_s + tile_off(mt * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8, bs));
                        mma_bf16_16816(c4, af, qb[kk][0], qb[kk][1]);
                    }
                }
                const int tok0 = tok_base + mt * 16 + gi, tok1 = tok0 + 8;
                sc[mi][0] = tok0 < L ? c4[0] * a.scale_log2 : -INFINITY;
                sc[mi][1] = tok0 < L ? c4[1] * a.scale_log2 : -INFINITY;
                sc[mi][2] = tok1 < L ? c4[2] * a.scale_log2 : -INFINITY;
                sc[mi][3] = tok1 < L ? c4[3] * a.scale_log2 : -INFINITY;
                bm0 = fmaxf(bm0, fmaxf(sc[mi][0], sc[mi][2]));
                bm1 = fmaxf(bm1, fmaxf(sc[mi][1], sc[mi][3]));
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
        }
        if (gi == 0) {
            S.red_max[warp][2 * t] = bm0;
            S.red_max[warp][2 * t + 1] = bm1;
        }
        named_barrier_sync(kBarConsumers, kAttnCW * 32);
        float mn0 = m_run0, mn1 = m_run1;
#pragma unroll
        for (int w = 0; w < kAttnCW; ++w) {
            mn0 = fmaxf(mn0, S.red_max[w][2 * t]);
            mn1 = fmaxf(mn1, S.red_max[w][2 * t + 1]);
        }
        const float al0 = exp2f(m_run0 - mn0), al1 = exp2f(m_run1 - mn1);  // 0 for the first block

        // ---- weights, rounded to bf16; their sums add the rounded values
        float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int mt = warp + kAttnCW * mi;
            if (mt < n_mt) {
                const __nv_bfloat16 p0 = __float2bfloat16_rn(exp2f(sc[mi][0] - mn0));
                const __nv_bfloat16 p1 = __float2bfloat16_rn(exp2f(sc[mi][1] - mn1));
                const __nv_bfloat16 p2 = __float2bfloat16_rn(exp2f(sc[mi][2] - mn0));
                const __nv_bfloat16 p3 = __float2bfloat16_rn(exp2f(sc[mi][3] - mn1));
                ps0 += __bfloat162float(p0) + __bfloat162float(p2);
                ps1 += __bfloat162float(p1) + __bfloat162float(p3);
                const int r = mt * 16 + gi;
                S.P[2 * t][r] = __bfloat16_as_ushort(p0);
                S.P[2 * t + 1][r] = __bfloat16_as_ushort(p1);
                S.P[2 * t][r + 8] = __bfloat16_as_ushort(p2);
                S.P[2 * t + 1][r + 8] = __bfloat16_as_ushort(p3);
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            ps0 += __shfl_xor_sync(0xffffffffu, ps0, o);
            ps1 += __shfl_xor_sync(0xffffffffu, ps1, o);
        }
        if (gi == 0) {
            S.red_sum[warp][2 * t] = ps0;
            S.red_sum[warp][2 * t + 1] = ps1;
        }
        named_barrier_sync(kBarConsumers, kAttnCW * 32);
        float bs0 = 0.0f, bs1 = 0.0f;
#pragma unroll
        for (int w = 0; w < kAttnCW; ++w) {
            bs0 += S.red_sum[w][2 * t];
            bs1 += S.red_sum[w][2 * t + 1];
        }
        l_run0 = l_run0 * al0 + bs0;
        l_run1 = l_run1 * al1 + bs1;
        m_run0 = mn0;
        m_run1 = mn1;

        // ---- O^T = alpha O^T + V^T P over this block's tokens
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            acc[x][0] *= al0;
            acc[x][1] *= al1;
            acc[x][2] *= al0;
            acc[x][3] *= al1;
        }
        if (ok) {
            for (int kt2 = 0; kt2 < n_mt; ++kt2) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&S.P[gi][kt2 * 16 + 2 * t]);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&S.P[gi][kt2 * 16 + 2 * t + 8]);
                const int tok = kt2 * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    if (x < mpw) {
                        const int d = (warp * mpw + x) * 16 + ((lane >> 3) & 1) * 8;
                        uint32_t af[4];
                        ldmatrix_x4_trans(af, vt_s + tile_off(tok, d, bs));
                        mma_bf16_16816(acc[x], af, b0, b1);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
    }

    // ---- this split's partial: max and sum per head, unnormalised O
    float *pml = a.part_ml + pidx * kAttnMaxGroup * 2;
    float *pacc = a.part_acc + pidx * kAttnMaxGroup * D;
    if (warp == 0 && gi == 0) {
        pml[(2 * t) * 2] = m_run0;
        pml[(2 * t) * 2 + 1] = l_run0;
        pml[(2 * t + 1) * 2] = m_run1;
        pml[(2 * t + 1) * 2 + 1] = l_run1;
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        if (x < mpw) {
            const int d0 = (warp * mpw + x) * 16 + gi;
            pacc[(2 * t) * D + d0] = acc[x][0];
            pacc[(2 * t + 1) * D + d0] = acc[x][1];
            pacc[(2 * t) * D + d0 + 8] = acc[x][2];
            pacc[(2 * t + 1) * D + d0 + 8] = acc[x][3];
        }
    }
}

// Merges the splits: o = sum_s 2^(m_s - m) O_s / sum_s 2^(m_s - m) l_s over the
// splits that saw tokens (a sequence without tokens gives zeros).  CTA
// (sequence x query head, 64-wide slice of D), 256 threads: thread (e, sg)
// takes float4 column e of the slice and splits sg, sg + 16, ...; it loads
// their (m, l) and partial O in one go (8 splits in flight), keeps a running
// max of its own and rescales as it goes, so the partials are read in a single
// pass.  The threads then agree on the common max, rescale, and the 16 groups'
// sums are added in a fixed order.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a)
{
    constexpr int kCols = 16, kGroups = 16, kBatch = 8;  // float4 columns, split groups, loads in flight
    __shared__ float4 part[kGroups][kCols];
    __shared__ float red_max[8], red_den[8];
    const int b = blockIdx.x / a.H_q, h = blockIdx.x - b * a.H_q;
    const int g = h / a.group, n = h - g * a.group;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = tid % kCols, sg = tid / kCols;
    pdl_trigger();
    pdl_wait();  // the split kernel is complete
    const size_t p0 = (static_cast<size_t>(b) * a.H_kv + g) * a.n_splits;
    const int S = a.n_splits, Q = a.D / 4, q = blockIdx.y * kCols + e;
    const bool act = q < Q;
    const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + (p0 * kAttnMaxGroup + n) * a.D) + (act ? q : 0);
    const float *mls = a.part_ml + (p0 * kAttnMaxGroup + n) * 2;
    const size_t stride4 = static_cast<size_t>(kAttnMaxGroup) * Q;
    float mt = -INFINITY, dt = 0.0f;
    float4 num = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int s0 = sg; s0 < S; s0 += kBatch * kGroups) {
        float4 v[kBatch];
        float2 ml[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int s = s0 + k * kGroups;
            ml[k] = s < S ? *reinterpret_cast<const float2 *>(mls + static_cast<size_t>(s) * kAttnMaxGroup * 2)
                          : make_float2(-INFINITY, 0.0f);
            v[k] = s < S && act ? src[static_cast<size_t>(s) * stride4] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        float bm = mt;
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (ml[k].y > 0.0f) bm = fmaxf(bm, ml[k].x);
        if (bm > -INFINITY) {
            const float c = exp2f(mt - bm);  // 0 while nothing was taken
            num.x *= c;
            num.y *= c;
            num.z *= c;
            num.w *= c;
            dt *= c;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (ml[k].y > 0.0f) {
                    const float w = exp2f(ml[k].x - bm);
                    num.x += w * v[k].x;
                    num.y += w * v[k].y;
                    num.z += w * v[k].z;
                    num.w += w * v[k].w;
                    dt += w * ml[k].y;
                }
            }
            mt = bm;
        }
    }
    float mx = mt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_max[warp] = mx;
    __syncthreads();
    mx = red_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red_max[w]);
    const float f = mt > -INFINITY ? exp2f(mt - mx) : 0.0f;
    num.x *= f;
    num.y *= f;
    num.z *= f;
    num.w *= f;
    part[sg][e] = num;
    // the sum of weights: the threads of column 0 hold every split once
    float den = e == 0 ? dt * f : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) red_den[warp] = den;
    __syncthreads();
    if (tid < kCols && act) {
        float4 t = part[0][tid];
#pragma unroll
        for (int g2 = 1; g2 < kGroups; ++g2) {
            t.x += part[g2][tid].x;
            t.y += part[g2][tid].y;
            t.z += part[g2][tid].z;
            t.w += part[g2][tid].w;
        }
        float dsum = red_den[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) dsum += red_den[w];
        const float r = dsum > 0.0f ? 1.0f / dsum : 0.0f;
        t.x *= r;
        t.y *= r;
        t.z *= r;
        t.w *= r;
        reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(b) * a.H_q + h) * a.D)[q] = t;
    }
}

}  // namespace

int attn_stages(int D, int bs) { return stages_for(D, bs); }

size_t attn_smem_bytes(int D, int bs)
{
    return 1024 + kAttnFixed + static_cast<size_t>(stages_for(D, bs)) * stage_bytes(D, bs);
}

cudaError_t launch_attn_decode(const AttnArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t stream)
{
    const size_t smem = attn_smem_bytes(a.D, a.bs);
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(attn_split_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_split_kernel, dim3(a.n_splits, a.H_kv, a.B), dim3(kAttnThreads), smem, stream, a, tmK, tmV);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_combine_kernel, dim3(a.B * a.H_q, (a.D + 63) / 64), dim3(256), 0, stream, a);
}

}  // namespace lily
