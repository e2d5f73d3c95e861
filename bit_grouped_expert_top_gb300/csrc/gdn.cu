// Gated DeltaNet scan with the recurrent state held in registers, for sm_103a.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br): 30 of the
// model's layers are Gated DeltaNet layers, a recurrence of fixed size
// (section "O modelo em tres formatos de carga"); their prefill scan keeps the
// state in registers (section "Prefill e decode: onde estao os ganhos").  The
// recurrence (gated delta rule), per value head h with key head
// hk = h / (H_v / H_k), state S (d_v x d_k), token t:
//   u_t = S_{t-1} k_t
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t u_t) k_t^T
//   o_t = scale S_t q_t
//
// GB300 design.  The rows of S evolve independently (row i needs only u_i,
// v_t[i] and the shared k_t, q_t), so the state is split by rows: CTA
// (16-row slice, value head), 2 threads per row, each holding d_k / 2 columns
// of its row in registers for the whole sequence (column groups of 4
// interleaved over the row's threads, so their shared-memory reads of k and q
// hit consecutive banks).  Each slice of the state is held twice, by two
// warps of different roles.  The recurrence warp carries the chain that
// feeds back (u_t = S_{t-1} k_t, beta_t (v_t - alpha_t u_t), the update) and
// leaves beta_t (v_t - alpha_t u_t) per token and row in shared memory; the
// output warp, one chunk behind, repeats the same updates from those values
// (bit-identical states) and forms o_t with q_t, work that nothing in the
// recurrence waits for.  The recurrence warp also copies the token inputs (q
// and k rows of the key head, this slice's 16 values of v, alpha and beta)
// into shared memory 32 tokens at a time with cp.async, two chunks ahead, and
// converts k and q to fp32 once per chunk for both roles; one block barrier
// per chunk hands a chunk from one role to the other.  The recurrence's token
// loop is pipelined (after the update with token t, the dot with k_{t+1});
// column pairs use the packed two-lane fp32 instructions.  Outputs of a chunk are
// collected in shared memory and written as 16-byte stores.  The sequential
// dependence through S makes the scan latency-bound: per token a chain of
// shared-memory loads, a few FMAs and a butterfly shuffle.
#include <cstdint>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kGdnRows = 16;      // state rows per CTA
constexpr int kGdnChunk = 32;     // tokens staged per buffer

template <int DK>
struct GdnStage {
    uint16_t k[kGdnChunk][DK];
    uint16_t q[kGdnChunk][DK];
    uint16_t v[kGdnChunk][kGdnRows];
    float alpha[kGdnChunk];
    float beta[kGdnChunk];
};

template <int DK>
struct GdnSmem {
    GdnStage<DK> st[2];              // bf16 inputs as copied (double buffered)
    float kf[2][kGdnChunk][DK];      // k and q in fp32, converted once for all rows; the
    float qf[2][kGdnChunk][DK];      // output warps read chunk c - 1 while chunk c is written
    float cc[2][kGdnChunk][kGdnRows];  // per token and row: beta (v - alpha u), from the recurrence warps
    float al[2][kGdnChunk];          // alpha of the chunk, for the output warps
    float o[kGdnChunk][kGdnRows];
};

__device__ __forceinline__ void cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Packed two-lane fp32 arithmetic (one instruction for two values).
__device__ __forceinline__ unsigned long long f2_bits(float2 v)
{
    return static_cast<unsigned long long>(__float_as_uint(v.x)) |
           (static_cast<unsigned long long>(__float_as_uint(v.y)) << 32);
}
__device__ __forceinline__ float2 f2_from(unsigned long long b)
{
    return make_float2(__uint_as_float(static_cast<uint32_t>(b)), __uint_as_float(static_cast<uint32_t>(b >> 32)));
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)  // a * b + c, each lane rounded once
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return f2_from(r);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_from(r);
}

// TPR threads per state row, each owning DK / TPR columns; 16 rows per CTA,
// held twice: by the recurrence warps and by the output warps.
template <int DK, int TPR>
__global__ void __launch_bounds__(2 * kGdnRows * TPR) gdn_scan_kernel(const GdnArgs a)
{
    constexpr int NR = kGdnRows * TPR;  // threads of one role (the block has two roles)
    constexpr int CPT = DK / TPR;       // state columns per thread
    extern __shared__ __align__(16) uint8_t gsm[];
    GdnSmem<DK> &S = *reinterpret_cast<GdnSmem<DK> *>(gsm);
    const int slice = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, rtid = tid % NR, r = rtid / TPR, cg = tid % TPR;
    const bool recur = tid < NR;  // recurrence warps; the others form the outputs
    const int hk = h / (a.H_v / a.H_k);
    const int row = slice * kGdnRows + r;
    const int T = a.T;

    pdl_trigger();
    pdl_wait();

    // Column ownership: thread cg of a row holds the 4-column groups m TPR + cg
    // (m < CPT / 4), so that a float4 step over a row's threads covers
    // consecutive addresses (no shared-memory bank conflicts).
    auto col = [&](int j) { return ((j >> 2) * TPR + cg) * 4 + (j & 3); };
    constexpr int NP = CPT / 2;  // column pairs per thread
    float2 st[NP];
    {
        const float *s0 = a.state_in ? a.state_in + (static_cast<size_t>(h) * a.d_v + row) * DK : nullptr;
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
            float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s0) v4 = *reinterpret_cast<const float4 *>(s0 + col(j));
            st[j / 2] = make_float2(v4.x, v4.y);
            st[j / 2 + 1] = make_float2(v4.z, v4.w);
        }
    }

    // recurrence threads: stage tokens [t0, t0 + n) into buffer b (one cp.async group)
    auto stage = [&](int b, int t0) {
        GdnStage<DK> &B = S.st[b];
        const int n = min(kGdnChunk, T - t0);
        constexpr int kPieces = DK * 2 / 16;  // 16-byte pieces of a q or k row
        for (int i = tid; i < n * kPieces; i += NR) {
            const int t = i / kPieces, p = i - t * kPieces;
            const size_t src = (static_cast<size_t>(t0 + t) * a.H_k + hk) * DK + p * 8;
            cp_async_16(&B.k[t][p * 8], a.k + src);
            cp_async_16(&B.q[t][p * 8], a.q + src);
        }
        for (int i = tid; i < n * 2; i += NR) {
            const int t = i >> 1, p = i & 1;
            cp_async_16(&B.v[t][p * 8], a.v + (static_cast<size_t>(t0 + t) * a.H_v + h) * a.d_v + slice * kGdnRows + p * 8);
        }
        for (int t = tid; t < n; t += NR) {
            cp_async_4(&B.alpha[t], a.alpha + static_cast<size_t>(t0 + t) * a.H_v + h);
            cp_async_4(&B.beta[t], a.beta + static_cast<size_t>(t0 + t) * a.H_v + h);
        }
        cp_async_commit();
    };

    // the row's partial sum over its TPR threads (consecutive lanes)
    auto row_sum = [](float x) {
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        return x;
    };
    auto load_row = [&](const float (*src)[DK], int t, float2(&dst)[NP]) {
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(&src[t][col(j)]);
            dst[j / 2] = make_float2(v4.x, v4.y);
            dst[j / 2 + 1] = make_float2(v4.z, v4.w);
        }
    };
    // four partial sums per dot, so each dependence chain is NP / 4 long; the
    // same order at every token, so a scan split between calls gives the same bits
    auto psum4 = [](const float2(&p)[4]) {
        return ((p[0].x + p[0].y) + (p[1].x + p[1].y)) + ((p[2].x + p[2].y) + (p[3].x + p[3].y));
    };

    // Chunk pipeline.  The recurrence threads stage the inputs two chunks ahead
    // and convert k and q of a chunk to fp32 before running its tokens; they
    // leave beta (v - alpha u) per token and row in shared memory.  The output
    // threads, one chunk behind, repeat the same state updates from those values
    // (the same bits) and form o_t with q_t, which nothing in the recurrence
    // waits for.  One barrier per iteration c: after it the recurrence on chunk
    // c and the outputs of chunk c - 1 are both done, so chunk c + 1 may be
    // converted into the buffers chunk c - 1 used, and the outputs of chunk c
    // may start.  One extra iteration lets the output threads finish.
    auto role_sync = [&]() {  // the NR threads of this thread's role
        if (recur)
            asm volatile("bar.sync 1, %0;" ::"n"(NR) : "memory");
        else
            asm volatile("bar.sync 2, %0;" ::"n"(NR) : "memory");
    };
    auto convert = [&](int c) {  // recurrence threads: k and q of chunk c to fp32, alpha copied
        const int b = c & 1, n = min(kGdnChunk, T - c * kGdnChunk);
        const GdnStage<DK> &B = S.st[b];
        for (int i = tid; i < n * DK / 8; i += NR) {
            const int t = i / (DK / 8), j = (i - t * (DK / 8)) * 8;
            const uint4 kw = *reinterpret_cast<const uint4 *>(&B.k[t][j]);
            const uint4 qw = *reinterpret_cast<const uint4 *>(&B.q[t][j]);
            float4 *kd = reinterpret_cast<float4 *>(&S.kf[b][t][j]), *qd = reinterpret_cast<float4 *>(&S.qf[b][t][j]);
            kd[0] = make_float4(__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xFFFF0000u),
                                __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xFFFF0000u));
            kd[1] = make_float4(__uint_as_float(kw.z << 16), __uint_as_float(kw.z & 0xFFFF0000u),
                                __uint_as_float(kw.w << 16), __uint_as_float(kw.w & 0xFFFF0000u));
            qd[0] = make_float4(__uint_as_float(qw.x << 16), __uint_as_float(qw.x & 0xFFFF0000u),
                                __uint_as_float(qw.y << 16), __uint_as_float(qw.y & 0xFFFF0000u));
            qd[1] = make_float4(__uint_as_float(qw.z << 16), __uint_as_float(qw.z & 0xFFFF0000u),
                                __uint_as_float(qw.w << 16), __uint_as_float(qw.w & 0xFFFF0000u));
        }
        for (int t = tid; t < n; t += NR) S.al[b][t] = B.alpha[t];
    };
    const int n_chunks = (T + kGdnChunk - 1) / kGdnChunk;
    if (recur && n_chunks > 0) {
        stage(0, 0);
        if (n_chunks > 1) {
            stage(1, kGdnChunk);
            cp_async_wait_1();  // chunk 0's group has landed (chunk 1's may still be in flight)
        } else {
            cp_async_wait_all();
        }
        role_sync();  // every thread's copies of chunk 0 are complete
        convert(0);
    }
    for (int c = 0; n_chunks > 0 && c <= n_chunks; ++c) {
        const int t0 = c * kGdnChunk, n = min(kGdnChunk, T - t0);
        const int b = c & 1;
        if (recur && c < n_chunks) {
            role_sync();  // chunk c's fp32 rows are complete
            // Token loop, pipelined: u_t = (S_{t-1} k_t)_row is ready on entry;
            // the update with token t is followed by the dot with k_{t+1}.  The
            // loop runs two tokens per trip so k_t and k_{t+1} swap register roles.
            const GdnStage<DK> &B = S.st[b];
            const float (*kf)[DK] = S.kf[b];
            float2 ka[NP], kb[NP];
            load_row(kf, 0, ka);
            float u;
            {
                float2 pa[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) pa[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NP; ++j) pa[j & 3] = ffma2(st[j], ka[j], pa[j & 3]);
                u = row_sum(psum4(pa));
            }
            auto step = [&](int t, const float2(&kc)[NP], float2(&kn)[NP]) {
                load_row(kf, t + 1 < n ? t + 1 : t, kn);
                const float al = B.alpha[t], be = B.beta[t];
                const float vr = __uint_as_float(static_cast<uint32_t>(B.v[t][r]) << 16);
                const float cc = be * (vr - al * u);
                if (cg == 0) S.cc[b][t][r] = cc;
                const float2 al2 = make_float2(al, al), cc2 = make_float2(cc, cc);
                float2 pa[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) pa[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    st[j] = ffma2(al2, st[j], fmul2(cc2, kc[j]));
                    pa[j & 3] = ffma2(st[j], kn[j], pa[j & 3]);
                }
                u = row_sum(psum4(pa));
            };
            int t = 0;
            for (; t + 1 < n; t += 2) {
                step(t, ka, kb);
                step(t + 1, kb, ka);
            }
            if (t < n) step(t, ka, kb);
            if (c + 2 < n_chunks) {
                role_sync();  // every recurrence thread is done with the staged chunk c
                stage(b, t0 + 2 * kGdnChunk);
            }
        } else if (!recur && c > 0) {
            // the previous chunk: S_t = alpha_t S_{t-1} + cc_t k_t^T, o_t = scale S_t q_t
            const int pb = b ^ 1, pn = min(kGdnChunk, T - (t0 - kGdnChunk));
            const float (*kf)[DK] = S.kf[pb];
            const float (*qf)[DK] = S.qf[pb];
#pragma unroll 2
            for (int t = 0; t < pn; ++t) {
                float2 kc[NP], qv[NP];
                load_row(kf, t, kc);
                load_row(qf, t, qv);
                const float al = S.al[pb][t], cc = S.cc[pb][t][r];
                const float2 al2 = make_float2(al, al), cc2 = make_float2(cc, cc);
                float2 oa[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) oa[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    st[j] = ffma2(al2, st[j], fmul2(cc2, kc[j]));
                    oa[j & 3] = ffma2(st[j], qv[j], oa[j & 3]);
                }
                const float o = row_sum(psum4(oa));
                if (cg == 0) S.o[t][r] = a.scale * o;
            }
            role_sync();  // the chunk's outputs are complete
            // per token 16 floats of this slice, four 16-byte stores
            const int pt0 = t0 - kGdnChunk;
            for (int i = tid - NR; i < pn * 4; i += NR) {
                const int t = i >> 2, p = i & 3;
                *reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(pt0 + t) * a.H_v + h) * a.d_v + slice * kGdnRows + p * 4) =
                    *reinterpret_cast<const float4 *>(&S.o[t][p * 4]);
            }
        }
        __syncthreads();
        if (recur && c + 1 < n_chunks) {
            // chunk c + 1 has landed: every group but the newest (chunk c + 2, if staged)
            if (c + 2 < n_chunks)
                cp_async_wait_1();
            else
                cp_async_wait_all();
            role_sync();  // every thread's copies of chunk c + 1 are complete
            convert(c + 1);
        }
    }
    if (recur) {
        float *so = a.state_out + (static_cast<size_t>(h) * a.d_v + row) * DK;
#pragma unroll
        for (int j = 0; j < CPT; j += 4)
            *reinterpret_cast<float4 *>(so + col(j)) = make_float4(st[j / 2].x, st[j / 2].y, st[j / 2 + 1].x, st[j / 2 + 1].y);
    }
}

}  // namespace

#ifndef LILY_GDN_TPR
#define LILY_GDN_TPR 2
#endif
constexpr int kGdnTPR = LILY_GDN_TPR;  // threads per state row

size_t gdn_smem_bytes(int d_k) { return d_k == 64 ? sizeof(GdnSmem<64>) : sizeof(GdnSmem<128>); }

template <int DK>
static cudaError_t launch_dk(const GdnArgs &a, cudaStream_t stream)
{
    const size_t smem = sizeof(GdnSmem<DK>);
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(gdn_scan_kernel<DK, kGdnTPR>), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(gdn_scan_kernel<DK, kGdnTPR>, dim3(a.d_v / kGdnRows, a.H_v), dim3(2 * kGdnRows * kGdnTPR), smem, stream, a);
}

cudaError_t launch_gdn_scan(const GdnArgs &a, cudaStream_t stream)
{
    return a.d_k == 64 ? launch_dk<64>(a, stream) : launch_dk<128>(a, stream);
}

}  // namespace lily
