// Device-side building blocks for the sm_103a kernels: inline PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor), cp.async, the 5th-generation tensor core
// (tcgen05.mma / tcgen05.ld with accumulators in tensor memory), bounded waits
// that report a timeout instead of hanging, the int4 -> fp16 dequantisation and
// the warp top-8 selection.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace lily {

// Device-detected error codes (same values as LILY_ERR_DEVICE_* in lily_moe.h).
constexpr int kErrDeviceTimeout = -6;
constexpr int kErrDeviceIndex = -7;
constexpr int kErrDeviceRange = -9;  // a finite value beyond the fp16 range of the expert GEMM operands

// Control block at the start of every workspace.
struct Ctrl {
    int status;             // sticky device status, 0 = OK
    unsigned int ticket;    // last-block-done counter of the routing kernel
    unsigned int ticket2;   // last-block-done counter of the decode router
    int pad[61];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

// Wall-clock bound of every pipeline spin-wait (nanoseconds).  A wait that
// exceeds it records kErrDeviceTimeout and gives up.
#ifndef LILY_WAIT_LIMIT_NS
#define LILY_WAIT_LIMIT_NS 2000000000ull
#endif
// Bound of the waits on a kernel's exit path, which wait for copies and
// tensor-core work already in flight before shared and tensor memory are
// given back.  It stays at 2 s in every build (a test build that shortens
// LILY_WAIT_LIMIT_NS keeps it), so nothing can still be writing when a CTA
// frees its tensor memory or exits.
#define LILY_DRAIN_LIMIT_NS 2000000000ull

__device__ __forceinline__ void record_error(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the waiting thread is parked by the
// hardware until the phase completes or about `hint_ns` nanoseconds pass, so a
// waiting warp does not take issue slots from working warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) when another role raised `abort_flag`, or after LILY_WAIT_LIMIT_NS, in
// which case it records kErrDeviceTimeout and raises `abort_flag`.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status)
{
    const uint32_t addr = smem_u32(bar);
    // with a suspend-time hint the thread wakes sooner after the phase completes
    // (measured median ~136 cycles against ~290 without one)
    if (mbar_try_wait_sleep(addr, parity, 20000u)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait_sleep(addr, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > LILY_WAIT_LIMIT_NS) {
            record_error(status, kErrDeviceTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

// Waits for two phases; both barriers are tested at once first, so that when
// both are already complete the thread pays one shared-memory round trip.
__device__ __forceinline__ bool mbar_wait2(uint64_t *bar0, uint32_t parity0, uint64_t *bar1, uint32_t parity1,
                                           volatile int *abort_flag, int *status)
{
    uint32_t ok0, ok1;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%2], %3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q, [%4], %5;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "selp.u32 %1, 1, 0, q;\n\t}"
        : "=r"(ok0), "=r"(ok1)
        : "r"(smem_u32(bar0)), "r"(parity0), "r"(smem_u32(bar1)), "r"(parity1)
        : "memory");
    if (ok0 && ok1) return true;
    return (ok0 || mbar_wait(bar0, parity0, abort_flag, status)) && (ok1 || mbar_wait(bar1, parity1, abort_flag, status));
}

// Programmatic dependent launch: this grid lets the next one start launching,
// and waits (before touching any global memory an earlier kernel of the stream
// reads or writes) until the preceding grid has completed and its memory is
// visible.  The waits chain, so after pdl_wait every earlier kernel is done.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled tensor load into shared memory; completion is signalled on `bar`
// as transaction bytes.  c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// ----------------------------------------------------------------- cp.async (16-byte gathers)
__device__ __forceinline__ void cp_async_16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Named barrier over `nthreads` threads (whole warps); the warp is reconverged
// first, as bar.sync is warp-aligned.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads)
{
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------- tcgen05 (UMMA + TMEM)
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs (type from idesc), fp32
// accumulate, both K-major.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A read from tensor memory (row m in lane m,
// two 16-bit K elements per 32-bit column), B K-major in shared memory.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 operand in the 128-byte
// swizzled layout: rows of 64 elements (128 B), 8-row atoms 1024 B apart.
// Bits: [0,14) start >> 4, [16,30) leading byte offset >> 4 (unused for this
// layout, set to 1), [32,46) stride byte offset >> 4 (1024 B between 8-row
// atoms), [46,48) descriptor version 1, [61,64) layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16 with an fp32 accumulator
// (bits 4-5 = 1).  A and B always share one input type, given by `ab_fmt`
// (0 = f16, 1 = bf16) in bits 7-9 and 10-12; both K-major (bits 15, 16 = 0);
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kFmtF16 = 0, kFmtBF16 = 1;
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t ab_fmt, int M, int N)
{
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 16 columns of 32-bit accumulator.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns store: thread i of the warp writes lane (base lane + i),
// columns [col, col + 32) from r[0..31].
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Two 6-bit e2m3 values (one per byte, low 6 bits) -> fp16 pair, low byte to
// the low half.  A byte holding a nibble q in its low 4 bits (sign 0, exponent
// bits 0 q3, mantissa q2 q1 q0) is exactly q / 8: subnormal q/8 for q < 8,
// (1 + (q-8)/8) for q >= 8.
__device__ __forceinline__ uint32_t cvt_e2m3x2_lo(uint32_t v)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e2m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(v));
    return r;
}
__device__ __forceinline__ uint32_t cvt_e2m3x2_hi(uint32_t v)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e2m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(v));
    return r;
}

// Eight packed 4-bit weights (element i in bits [4i, 4i+4)) -> eight fp16
// weights w_i = q_i * s + b, each rounded once: the nibbles are spread one per
// byte, converted to q/8 exactly (e2m3), then fma.rn.f16x2(q/8, 8 s, b), which
// equals fma(q, s, b) because 8 s is exact.  `s8` = 8 s.  Output K order within
// the group of 8: (0,2, 4,6, 1,3, 5,7); the other GEMM operand must use the same
// order (kperm8_e2m3).
__device__ __forceinline__ uint4 dequant8_f16_e2m3(uint32_t v, __half2 s8, __half2 b2)
{
    const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;  // nibbles 0,2,4,6 / 1,3,5,7
    const uint32_t q02 = cvt_e2m3x2_lo(lo), q46 = cvt_e2m3x2_hi(lo);
    const uint32_t q13 = cvt_e2m3x2_lo(hi), q57 = cvt_e2m3x2_hi(hi);
    __half2 f0 = __hfma2(*reinterpret_cast<const __half2 *>(&q02), s8, b2);
    __half2 f1 = __hfma2(*reinterpret_cast<const __half2 *>(&q46), s8, b2);
    __half2 f2 = __hfma2(*reinterpret_cast<const __half2 *>(&q13), s8, b2);
    __half2 f3 = __hfma2(*reinterpret_cast<const __half2 *>(&q57), s8, b2);
    return make_uint4(*reinterpret_cast<uint32_t *>(&f0), *reinterpret_cast<uint32_t *>(&f1),
                      *reinterpret_cast<uint32_t *>(&f2), *reinterpret_cast<uint32_t *>(&f3));
}

// Position of logical K index k in the order used by dequant8_f16_e2m3: inside
// each group of 8, even elements j at j/2, odd ones at 4 + j/2.
__host__ __device__ __forceinline__ int kperm8_e2m3(int k)
{
    const int j = k & 7;
    return (k & ~7) | ((j >> 1) + ((j & 1) << 2));
}

// True if either half of a packed fp16 pair is infinite: a finite input
// (bf16 x, or the fp32 SwiGLU product h) at or beyond 65520 in magnitude
// rounds to infinity when it is converted to an fp16 GEMM operand.
__device__ __forceinline__ bool f16x2_has_inf(uint32_t v)
{
    const uint32_t a = v & 0x7FFF7FFFu;
    return ((a & 0xFFFFu) == 0x7C00u) | ((a >> 16) == 0x7C00u);
}

// bf16 bit pattern -> fp16 pair (value converted with round-to-nearest).
__device__ __forceinline__ __half2 half2_from_bf16_bits(uint16_t bits)
{
    const __half h = __float2half_rn(__uint_as_float(static_cast<uint32_t>(bits) << 16));
    return __halves2half2(h, h);
}

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Asynchronous prefetch of `bytes` (multiple of 16, 16-byte aligned address)
// of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-bit values [g0, g0 + 8) of a row of n values, packed two per word (zero
// past the end).  `vec` allows one 16-byte load (row 16-byte aligned, n % 8 == 0).
__device__ __forceinline__ uint4 load_groups8(const uint16_t *row, int g0, int n, bool vec)
{
    if (g0 >= n) return make_uint4(0u, 0u, 0u, 0u);
    if (vec) return __ldg(reinterpret_cast<const uint4 *>(row + g0));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (g0 + j < n) w[j >> 1] |= static_cast<uint32_t>(__ldg(row + g0 + j)) << (16 * (j & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Value j (0..3) of four 16-bit values packed two per word.
__device__ __forceinline__ uint16_t pick16x4(const uint2 v, int j)
{
    const uint32_t w = (j & 2) ? v.y : v.x;
    return static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// silu(z) = z sigmoid(z), with sigmoid(z) = (1 + tanh(z / 2)) / 2 and the
// hardware tanh approximation (one special-function op per value; its error,
// about 2^-11 of |tanh|, stays near the fp16 rounding of the result).
__device__ __forceinline__ float tanh_approx(float v)
{
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float silu_f(float z)
{
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_approx(hz), hz);
}

// ----------------------------------------------------------------- top-8 of 256 (one warp)
// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_order_key(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0, so equal values tie
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of float_order_key.
__device__ __forceinline__ float float_from_order_key(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Selects the 8 largest of 256 fp32 logits given as 8 per lane (lane l holds
// logits 8l..8l+7), ordered by descending logit with the lower expert index
// first among equal logits, and their renormalised softmax weights
// w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0).  Lane j < 8 receives slot j.
// Eight rounds on 32-bit order-preserving keys: each lane takes the maximum of
// its remaining keys, one warp reduction gives the round's maximum, and the
// lowest lane holding it wins (lane l holds the lower indices 8l..8l+7); the
// winner takes out its first key equal to the maximum (its lowest index among
// equal logits).  Key 0 marks a taken slot: it is below the key of every
// finite logit, -inf included.
__device__ __forceinline__ void warp_top8_keys(const float (&lv)[8], int lane, int &sel_e, float &sel_w)
{
    uint32_t key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) key[j] = float_order_key(lv[j]);
    uint32_t top = 0u, mine = 0u;
    int mine_e = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const uint32_t lm = max(max(max(key[0], key[1]), max(key[2], key[3])),
                                max(max(key[4], key[5]), max(key[6], key[7])));
        const uint32_t wm = __reduce_max_sync(0xffffffffu, lm);
        const int win = __ffs(__ballot_sync(0xffffffffu, lm == wm)) - 1;
        int pos = 7;
#pragma unroll
        for (int j = 6; j >= 0; --j)
            if (key[j] == wm) pos = j;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (lane == win && j == pos) key[j] = 0u;
        const int wpos = __shfl_sync(0xffffffffu, pos, win);
        if (r == 0) top = wm;
        if (lane == r) {
            mine = wm;
            mine_e = win * 8 + wpos;
        }
    }
    sel_e = mine_e;
    const float sel_v = float_from_order_key(mine);
    const float vmax = float_from_order_key(top);
    const float ex = lane < 8 ? expf(sel_v - vmax) : 0.0f;
    float den = ex;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    sel_w = ex / den;
}

}  // namespace lily
