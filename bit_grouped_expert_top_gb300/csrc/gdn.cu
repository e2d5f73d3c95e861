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
// (16-row slice, value head), 128 threads, eight threads per row, each owning
// d_k / 8 columns of its row in registers for the whole sequence.  Per token a
// thread does its part of S k, the eight partial sums meet in three
// butterfly shuffles, then the rank-1 update of its columns and its part of
// S q (three more shuffles).  The token inputs (q and k rows of the key head,
// this slice's 16 values of v, alpha and beta) are staged in shared memory
// 64 tokens at a time with cp.async, double buffered, so the scan never waits
// on global memory; outputs of a chunk are collected in shared memory and
// written as 16-byte stores.  The sequential dependence through S makes the
// scan latency- and ALU-bound, not bandwidth-bound.
#include <cstdint>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kGdnThreads = 128;
constexpr int kGdnRows = 16;      // state rows per CTA
constexpr int kGdnChunk = 64;     // tokens staged per buffer

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
    GdnStage<DK> st[2];
    float o[kGdnChunk][kGdnRows];
};

__device__ __forceinline__ void cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// 8 consecutive bf16 values (16 bytes of shared memory) -> floats
__device__ __forceinline__ void bf16x8_to_f32(const uint16_t *p, float *f)
{
    const uint4 w = *reinterpret_cast<const uint4 *>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

template <int DK>
__global__ void __launch_bounds__(kGdnThreads) gdn_scan_kernel(const GdnArgs a)
{
    constexpr int CPT = DK / 8;  // state columns per thread
    extern __shared__ __align__(16) uint8_t gsm[];
    GdnSmem<DK> &S = *reinterpret_cast<GdnSmem<DK> *>(gsm);
    const int slice = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, r = tid >> 3, cg = tid & 7;
    const int hk = h / (a.H_v / a.H_k);
    const int row = slice * kGdnRows + r;
    const int T = a.T;

    pdl_trigger();
    pdl_wait();

    float st[CPT];
    {
        const float *s0 = a.state_in ? a.state_in + (static_cast<size_t>(h) * a.d_v + row) * DK + cg * CPT : nullptr;
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
            float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s0) v4 = *reinterpret_cast<const float4 *>(s0 + j);
            st[j] = v4.x;
            st[j + 1] = v4.y;
            st[j + 2] = v4.z;
            st[j + 3] = v4.w;
        }
    }

    // stage tokens [t0, t0 + n) into buffer b (one cp.async group)
    auto stage = [&](int b, int t0) {
        GdnStage<DK> &B = S.st[b];
        const int n = min(kGdnChunk, T - t0);
        constexpr int kPieces = DK * 2 / 16;  // 16-byte pieces of a q or k row
        for (int i = tid; i < n * kPieces; i += kGdnThreads) {
            const int t = i / kPieces, p = i - t * kPieces;
            const size_t src = (static_cast<size_t>(t0 + t) * a.H_k + hk) * DK + p * 8;
            cp_async_16(&B.k[t][p * 8], a.k + src);
            cp_async_16(&B.q[t][p * 8], a.q + src);
        }
        for (int i = tid; i < n * 2; i += kGdnThreads) {
            const int t = i >> 1, p = i & 1;
            cp_async_16(&B.v[t][p * 8], a.v + (static_cast<size_t>(t0 + t) * a.H_v + h) * a.d_v + slice * kGdnRows + p * 8);
        }
        for (int t = tid; t < n; t += kGdnThreads) {
            cp_async_4(&B.alpha[t], a.alpha + static_cast<size_t>(t0 + t) * a.H_v + h);
            cp_async_4(&B.beta[t], a.beta + static_cast<size_t>(t0 + t) * a.H_v + h);
        }
        cp_async_commit();
    };

    const int n_chunks = (T + kGdnChunk - 1) / kGdnChunk;
    if (n_chunks > 0) stage(0, 0);
    for (int c = 0; c < n_chunks; ++c) {
        const int t0 = c * kGdnChunk, n = min(kGdnChunk, T - t0);
        if (c + 1 < n_chunks) {
            stage((c + 1) & 1, t0 + kGdnChunk);
            cp_async_wait_1();  // this chunk's group has landed (the next one may still be in flight)
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const GdnStage<DK> &B = S.st[c & 1];
        for (int t = 0; t < n; ++t) {
            float kf[CPT];
#pragma unroll
            for (int j = 0; j < CPT; j += 8) bf16x8_to_f32(&B.k[t][cg * CPT + j], kf + j);
            // u = (S k)_row: four independent partial chains, then the 8 threads of the row
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < CPT; ++j) p[j & 3] = fmaf(st[j], kf[j], p[j & 3]);
            float u = (p[0] + p[1]) + (p[2] + p[3]);
            u += __shfl_xor_sync(0xffffffffu, u, 1);
            u += __shfl_xor_sync(0xffffffffu, u, 2);
            u += __shfl_xor_sync(0xffffffffu, u, 4);
            const float al = B.alpha[t], be = B.beta[t];
            const float vr = __uint_as_float(static_cast<uint32_t>(B.v[t][r]) << 16);
            const float cc = be * (vr - al * u);
            float qf[CPT];
#pragma unroll
            for (int j = 0; j < CPT; j += 8) bf16x8_to_f32(&B.q[t][cg * CPT + j], qf + j);
            float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                st[j] = fmaf(al, st[j], cc * kf[j]);
                o4[j & 3] = fmaf(st[j], qf[j], o4[j & 3]);
            }
            float o = (o4[0] + o4[1]) + (o4[2] + o4[3]);
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            o += __shfl_xor_sync(0xffffffffu, o, 2);
            o += __shfl_xor_sync(0xffffffffu, o, 4);
            if (cg == 0) S.o[t][r] = a.scale * o;
        }
        __syncthreads();
        // the chunk's outputs: per token 16 floats of this slice, four 16-byte stores
        for (int i = tid; i < n * 4; i += kGdnThreads) {
            const int t = i >> 2, p = i & 3;
            *reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(t0 + t) * a.H_v + h) * a.d_v + slice * kGdnRows + p * 4) =
                *reinterpret_cast<const float4 *>(&S.o[t][p * 4]);
        }
        // the buffer just read is restaged two chunks later, after the barrier above
    }
    float *so = a.state_out + (static_cast<size_t>(h) * a.d_v + row) * DK + cg * CPT;
#pragma unroll
    for (int j = 0; j < CPT; j += 4) *reinterpret_cast<float4 *>(so + j) = make_float4(st[j], st[j + 1], st[j + 2], st[j + 3]);
}

}  // namespace

size_t gdn_smem_bytes(int d_k) { return d_k == 64 ? sizeof(GdnSmem<64>) : sizeof(GdnSmem<128>); }

cudaError_t launch_gdn_scan(const GdnArgs &a, cudaStream_t stream)
{
    const dim3 grid(a.d_v / kGdnRows, a.H_v);
    const size_t smem = gdn_smem_bytes(a.d_k);
    if (a.d_k == 64) {
        cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(gdn_scan_kernel<64>), static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        return launch_pdl(gdn_scan_kernel<64>, grid, dim3(kGdnThreads), smem, stream, a);
    }
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(gdn_scan_kernel<128>), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(gdn_scan_kernel<128>, grid, dim3(kGdnThreads), smem, stream, a);
}

}  // namespace lily
