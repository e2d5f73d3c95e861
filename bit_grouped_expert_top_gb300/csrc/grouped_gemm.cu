// Persistent, warp-specialised tcgen05 grouped GEMM for the MoE layer on sm_103a.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br, section "Prefill e
// decode: onde estao os ganhos"): the expert GEMMs run over uneven per-expert
// token groups, and the 4-bit group-64 affine weights are rebuilt one tile at a
// time inside the GEMM, held on chip, with FP32 accumulation.  The page rebuilds
// to bf16 because its tensor ops take bf16; tcgen05 takes fp16 at the same
// rate and fp16 rounds the rebuilt weight 8x more finely, so the expert GEMMs
// here run on fp16 operands (x converted once; h written as fp16).  The router
// GEMM stays bf16 (its inputs are bf16 and the products are exact in fp32).
//
// GB300 design.  The weights take the UMMA M side (128 rows per tile, two
// tiles per work unit sharing one B operand: gate+up rows of the same
// intermediate slice, or two adjacent 128-row slices of the down projection)
// and the tokens of one block-map entry take the N side (N = rows rounded up
// to 16, at most 128), so small expert groups waste little tensor work.
// One CTA per SM loops over work units:
//   warp 0        A-side producer: TMA of the packed int4 tiles (expert modes)
//                 or of the bf16 router weights;
//   warp 2        B producer: 2-D TMA of contiguous token rows: x (router),
//                 x in routing order (gate/up; written by the prep kernel),
//                 h (down);
//   warps 1, 3    tcgen05.mma issuers, one thread each: warp 1 the first
//                 weight tile's accumulator, warp 3 the second's (one thread
//                 alone cannot issue the MMAs as fast as the tensor core runs
//                 them while the dequantisers share its SM sub-partition);
//                 warp 1 also allocates TMEM;
//   warps 4..11   dequantisers (expert modes): int4 -> fp16, one row per
//                 thread, each warp 32 rows of one matrix on its own pace,
//                 written to tensor memory with tcgen05.st; the MMA reads A
//                 from tensor memory (TS form);
//   warps 12..19  epilogue: tcgen05.ld from TMEM, then per mode the router
//                 logits (+bias), SwiGLU into h (fp16), or the down projection
//                 scaled by the routing weight and added (red.global.add.f32)
//                 into token order; in gate/up mode they first zero this CTA's
//                 slice of `out` (for the down projection) while the first
//                 unit's MMAs run.
// The K loop runs in blocks of four 64-wide k-steps (one raw int4 stage, one
// pass over the 4-stage tensor-memory A ring), so every ring slot and phase
// parity inside a block is a compile-time constant and the single-thread roles
// spend few instructions per k-step.  K is padded up to a multiple of 256: the
// copies read zeros past the end of K and the padded weights rebuild to zero.
// Every wait is bounded; on timeout the kernel records the error, drains its
// in-flight copies and tensor-core work, frees TMEM and returns.
#include <algorithm>
#include <cstddef>
#include <cstdio>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kThreads = 640;  // 20 warps: 4 producer/MMA, 8 dequant, 8 epilogue
constexpr int kBlk = 4;        // k-steps per block: one raw stage, one tensor-memory A ring cycle
constexpr int kRStages = 2;    // raw int4 ring (TMA), one block per stage
constexpr int kBStages = 4;    // B ring in the dedicated buffers (router)
constexpr int kBSlotBars = 4;  // B ring slots (router: 4 x 1 k-step; expert modes: 4 x 2 k-steps, the last
                               // two in the shared-memory A buffers they do not use)
constexpr int kAStages = 2;    // shared-memory A ring (bf16 router weights by TMA)
constexpr int kTAStages = 2;   // tensor-memory A ring (expert modes: 2 stages of 2 k-steps)
constexpr int kRouterAStages = 4;  // router: bf16 A ring in `a` and `raw` (which it does not otherwise use)
constexpr int kABars = 4;          // full_a / empty_a barriers: max(kTAStages, kRouterAStages)
constexpr int kTileM = 128;
constexpr int kBK = 64;        // one quantisation group, one 128-byte swizzle row
constexpr int kTileN = 128;
constexpr int kABytes = kTileM * kBK * 2;    // 16 KB of 16-bit elements
constexpr int kBBytes = kTileN * kBK * 2;    // 16 KB of 16-bit elements
constexpr int kRawRow = kBlk * kBK / 2;      // 128 B of packed int4 per row per raw stage
constexpr int kRawBytes = kTileM * kRawRow;  // 16 KB int4 per matrix
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulators at [0, 256) per buffer (router: two buffers, [0, 512));
// expert modes: one accumulator buffer and the A ring at [256, 512): stage h at
// 256 + 128 h, matrix m at + 64 m, k-step j of the stage at + 32 j.
constexpr uint32_t kTmemAOffset = 256;
constexpr int kBarEpilogue = 3;  // named barrier id
constexpr int kIssuers = 2;      // MMA-issuing threads (warps 1 and 3), one per weight tile
static_assert(kBStages == kBlk && kAStages == 2 && kTAStages == 2, "ring slots are compile-time within a block");

struct __align__(1024) Smem {
    uint8_t b[kBStages][kBBytes];         // B ring; expert modes continue into `a`
    uint8_t a[kAStages][2][kABytes];      // router: bf16 A ring; expert modes: B stages 4..7
    uint8_t raw[kRStages][2][kRawBytes];
    uint64_t full_r[kRStages], empty_r[kRStages];
    uint64_t full_b[kBSlotBars], empty_b[kBSlotBars];
    uint64_t full_a[kABars], empty_a[kABars];
    uint64_t full_acc[2], empty_acc[2];
    uint64_t drain;
#ifdef LILY_TEST_STALL_T
    uint64_t never;        // test builds only: a barrier nothing arrives on
#endif
    uint32_t tmem_base;
    int abort_flag;
    int ep_go;             // epilogue's wait result, published by its waiting thread
    int ep_tok[kTileN];    // epilogue: token of each column (down)
    float ep_w[kTileN];    // epilogue: routing weight of each column (down)
};
static_assert(sizeof(Smem) + 1024 <= 200 * 1024, "shared memory budget of one CTA");
static_assert(offsetof(Smem, a) == offsetof(Smem, b) + sizeof(Smem::b) &&
                  sizeof(Smem::a) == sizeof(Smem::b),
              "expert-mode B slots 2..3 continue the B ring in the A buffers");
static_assert(offsetof(Smem, raw) == offsetof(Smem, a) + sizeof(Smem::a) && sizeof(Smem::raw) == sizeof(Smem::a) &&
                  kRouterAStages * 2 * kABytes == sizeof(Smem::a) + sizeof(Smem::raw),
              "router A stages 2..3 continue the A ring in the raw buffers");

struct Unit {
    int e, p0, rows, n_mma, mt;
    bool shared;
};

template <int MODE>
__device__ __forceinline__ Unit unit_info(const GemmArgs &g, int tile, int n_routed)
{
    Unit u;
    const int b = tile / g.m_tiles;
    u.mt = tile - b * g.m_tiles;
    if (MODE != kModeRouter && b < n_routed) {
        const int *bm = g.block_map + 3 * b;
        u.e = bm[0];
        u.p0 = bm[1];
        u.rows = bm[2];
        u.shared = false;
        if (u.e < 0 || u.e >= g.E || u.p0 < 0 || u.rows < 1 || u.rows > g.bm || u.p0 + u.rows > g.T * g.top_k) {
            record_error(&g.ctrl->status, kErrDeviceIndex);
            u.rows = 0;
        }
    } else {
        const int sb = (MODE == kModeRouter) ? b : b - n_routed;
        u.e = -1;
        u.p0 = sb * g.bm;
        u.rows = min(g.bm, g.T - u.p0);
        u.shared = true;
    }
    u.n_mma = (u.rows + 15) & ~15;
    return u;
}

// First weight row of the two 128-row A tiles of a unit.
template <int MODE>
__device__ __forceinline__ void a_rows(const GemmArgs &g, const Unit &u, int &r0, int &r1)
{
    if (MODE == kModeRouter) {
        r0 = 0;
        r1 = kTileM;
    } else if (MODE == kModeGateUp) {
        r0 = (u.shared ? 0 : u.e * g.I) + u.mt * kTileM;
        r1 = r0;
    } else {
        r0 = (u.shared ? 0 : u.e * g.d) + u.mt * 2 * kTileM;
        r1 = r0 + kTileM;
    }
}

// Wait used on the exit path: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, int *status)
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

// 64-bit shared-memory descriptor from its two halves (the low half holds the
// start address >> 4, so a byte offset o within 256 KB adds o >> 4 to it).
__device__ __forceinline__ uint64_t desc64(uint32_t lo, uint32_t hi)
{
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Waits for the last min(issued, depth) phases of a ring's full barriers.
__device__ __forceinline__ void drain_ring(uint64_t *full, int depth, int issued, int *status)
{
    const int last = issued < depth ? issued : depth;
    for (int i = 1; i <= last; ++i) {
        const int step = issued - i;
        drain_wait(&full[step % depth], (step / depth) & 1, status);
    }
}

// B slot i of SS k-steps: slots continue from the dedicated buffers into the
// shared-memory A buffers (expert modes: 4 slots of 2 k-steps = 128 KB).
template <int SS>
__device__ __forceinline__ uint8_t *b_stage(Smem &S, int i)
{
    return reinterpret_cast<uint8_t *>(&S) + offsetof(Smem, b) + static_cast<size_t>(i) * SS * kBBytes;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmSA0, const __grid_constant__ CUtensorMap tmSA1)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int *status = &g.ctrl->status;
    constexpr bool dequant_mode = MODE != kModeRouter;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(&S.full_r[s], 1);
            mbar_init(&S.empty_r[s], 8);  // the eight dequantiser warps
        }
        for (int s = 0; s < kBSlotBars; ++s) {
            mbar_init(&S.full_b[s], 1);
            mbar_init(&S.empty_b[s], kIssuers);  // one commit per MMA issuer
        }
        for (int s = 0; s < kABars; ++s) {
            mbar_init(&S.full_a[s], dequant_mode ? 8 : 1);  // dequantiser warps / router TMA
            mbar_init(&S.empty_a[s], kIssuers);  // router only
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.full_acc[s], kIssuers);
            mbar_init(&S.empty_acc[s], 8);
        }
        mbar_init(&S.drain, kIssuers);
#ifdef LILY_TEST_STALL_T
        mbar_init(&S.never, 1);
#endif
        S.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA0);
        prefetch_tmap(&tmA1);
        prefetch_tmap(&tmB);
        if (dequant_mode) {
            prefetch_tmap(&tmSA0);
            prefetch_tmap(&tmSA1);
        }
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int *abort_flag = &S.abort_flag;
    // the setup above overlaps the previous kernel's tail; global memory only from here
    pdl_trigger();
    pdl_wait();
    if (MODE == kModeRouter && threadIdx.x == 0 && blockIdx.x == 0) g.ctrl->ticket = 0u;  // reset for the routing kernels

    int n_routed = 0;
    if (MODE != kModeRouter) {
        n_routed = *g.n_blocks;
        if (n_routed < 0 || n_routed > g.n_routed_max) {
            if (threadIdx.x == 0) record_error(status, kErrDeviceIndex);
            n_routed = 0;
        }
    }
    const int KS = (MODE == kModeRouter && g.ksplit > 1) ? g.ksplit : 1;  // router K splits
    const int total_tiles = (n_routed + g.n_shared_blocks) * g.m_tiles * KS;
    const int KB = g.KT / kBlk;  // blocks of four k-steps per unit (K padded)
    // tile -> unit ut (router: its block) and the unit's K blocks [kb0, kb1)
    auto k_range = [&](int tile, int &ut, int &kb0, int &kb1) {
        ut = tile / KS;
        const int ks = tile - ut * KS;
        kb0 = ks * KB / KS;
        kb1 = (ks + 1) * KB / KS;
    };

    // Abort handling: a bounded wait that gives up raises abort_flag; every
    // later wait then returns at once.  Single-thread roles leave their loops;
    // multi-warp groups keep walking their loops (skipping work) so that every
    // thread still reaches every named barrier of its group.
    //
    // Ring bookkeeping: `blk` counts blocks of four k-steps over all units of
    // this CTA; a block holds SPB stages of SS k-steps (expert modes: 2 stages
    // of 2 k-steps; router: 4 stages of 1).  Raw stage = blk % 2 (phase
    // (blk / 2) % 2).  Expert modes: tensor-memory A stage h (phase blk % 2),
    // free again once the MMAs of the same stage one block back completed,
    // i.e. B slot 2 ((blk - 1) % 2) + h (phase ((blk - 1) / 2) % 2); B slot
    // 2 (blk % 2) + h (phase (blk / 2) % 2).  Router: shared-memory A stage
    // = k-step within the block (phase blk % 2; four stages, the last two in the
    // raw buffers); B slot = k-step (phase blk % 2).
    constexpr int SS = dequant_mode ? 2 : 1;  // k-steps per stage
    constexpr int SPB = kBlk / SS;            // stages per block
    // B slots: router 4 x 1 k-step, expert modes 4 x 2 k-steps (two blocks per
    // ring cycle)
    constexpr int NSLOT = 4;
    constexpr int CYC = NSLOT / SPB;  // blocks per B ring cycle (1 or 2)
    if (warp == 0) {
        // ------------------------------------------------ A-side producer (one thread)
        if (lane == 0) {
            int blk = 0, issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                int ut, kb0, kb1;
                k_range(tile, ut, kb0, kb1);
                const Unit u = unit_info<MODE>(g, ut, n_routed);
                if (u.rows <= 0) continue;
                int r0, r1;
                a_rows<MODE>(g, u, r0, r1);
                const CUtensorMap *mA0 = u.shared ? &tmSA0 : &tmA0;
                const CUtensorMap *mA1 = u.shared ? &tmSA1 : &tmA1;
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++blk) {
                    if (dequant_mode) {
                        // one raw stage: 4 k-steps = 128 contiguous bytes of each row
                        const int rs = blk & 1;
                        if (!mbar_wait(&S.empty_r[rs], ((blk >> 1) & 1) ^ 1, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&S.full_r[rs], 2 * kRawBytes);
                        tma_load_2d(S.raw[rs][0], mA0, &S.full_r[rs], kb * kRawRow, r0);
                        tma_load_2d(S.raw[rs][1], mA1, &S.full_r[rs], kb * kRawRow, r1);
                        ++issued;
                    } else {
                        // one ring cycle per block: stage jr (k-step jr of the block), phase blk % 2
#pragma unroll
                        for (int jr = 0; jr < kBlk; ++jr) {
                            const int as = jr;
                            if (!mbar_wait(&S.empty_a[as], (blk & 1) ^ 1, abort_flag, status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&S.full_a[as], 2 * kABytes);
                            const int kc = (kb * kBlk + jr) * kBK;
                            uint8_t *dst = &S.a[0][0][0] + static_cast<size_t>(as) * 2 * kABytes;
                            tma_load_2d(dst, &tmA0, &S.full_a[as], kc, r0);
                            tma_load_2d(dst + kABytes, &tmA0, &S.full_a[as], kc, r1);
                            ++issued;
                        }
                    }
                }
            }
            // Exit: no copy into this CTA's shared memory may still be in flight.
            if (dequant_mode)
                drain_ring(S.full_r, kRStages, issued, status);
            else
                drain_ring(S.full_a, kRouterAStages, issued, status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ B producer (token rows)
        if (lane == 0) {
            // contiguous rows (x for the router; x in routing order for gate/up; h for
            // the down projection): one 2-D TMA per k-step
            int blk = 0, issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                int ut, kb0, kb1;
                k_range(tile, ut, kb0, kb1);
                const Unit u = unit_info<MODE>(g, ut, n_routed);
                if (u.rows <= 0) continue;
                // expert modes: routed rows in routing order, then the shared expert's
                // rows (token order) after the T * top_k routed rows
                const int b_row0 = (dequant_mode && u.shared) ? g.T * g.top_k + u.p0 : u.p0;
                if (dequant_mode) {
                    // warm L2 with the B rows of this CTA's next unit (contiguous rows)
                    const int nt = tile + gridDim.x;
                    if (nt < total_tiles) {
                        const Unit un = unit_info<MODE>(g, nt, n_routed);
                        if (un.rows > 0) {
                            const size_t row0 = un.shared ? static_cast<size_t>(g.T) * g.top_k + un.p0 : un.p0;
                            const __half *src = MODE == kModeGateUp ? g.xs : g.h;
                            bulk_prefetch_l2(src + row0 * g.K, static_cast<uint32_t>(un.rows) * g.K * 2u);
                        }
                    }
                }
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++blk) {
                    const uint32_t bpar = (CYC == 2 ? (blk >> 1) : blk) & 1;
#pragma unroll
                    for (int h = 0; h < SPB; ++h) {
                        const int bs = (CYC == 2 ? (blk & 1) : 0) * SPB + h;
                        if (!mbar_wait(&S.empty_b[bs], bpar ^ 1, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&S.full_b[bs], SS * kBBytes);
#pragma unroll
                        for (int j = 0; j < SS; ++j)
                            tma_load_2d(b_stage<SS>(S, bs) + j * kBBytes, &tmB, &S.full_b[bs], (kb * kBlk + h * SS + j) * kBK,
                                        b_row0);
                        ++issued;
                    }
                }
            }
            drain_ring(S.full_b, NSLOT, issued, status);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issuers (one thread each)
        // Thread of warp 1: the first weight tile (accumulator d0); warp 3: the
        // second (d1).  Each accumulator has one issuer, so its MMAs keep their
        // order; both wait for the same stages and both commit every release.
        const int mat = warp == 1 ? 0 : 1;
        if (lane == 0) {
            int blk = 0, ab = 0;
            uint32_t acc_ph = 0;
            bool ok = true;
            const uint32_t fmt = dequant_mode ? kFmtF16 : kFmtBF16;
            const int n_acc = dequant_mode ? 1 : 2;  // accumulator buffers in TMEM
            const uint64_t bd0 = sdesc_sw128(smem_u32(b_stage<SS>(S, 0)));
            const uint32_t b_lo = static_cast<uint32_t>(bd0), b_hi = static_cast<uint32_t>(bd0 >> 32);
            const uint64_t ad0 = sdesc_sw128(smem_u32(S.a[0][0]));
            const uint32_t a_lo = static_cast<uint32_t>(ad0), a_hi = static_cast<uint32_t>(ad0 >> 32);
            const uint32_t ta = tmem_base + kTmemAOffset;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                int ut, kb0, kb1;
                k_range(tile, ut, kb0, kb1);
                const Unit u = unit_info<MODE>(g, ut, n_routed);
                if (u.rows <= 0) continue;
                if (!mbar_wait(&S.empty_acc[ab], acc_ph ^ 1, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t idesc = idesc_f32acc(fmt, kTileM, u.n_mma);
                const uint32_t dm = tmem_base + static_cast<uint32_t>(ab * 2 * kTileM + mat * kTileM);
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++blk) {
                    const uint32_t bpar = (CYC == 2 ? (blk >> 1) : blk) & 1;
#pragma unroll
                    for (int h = 0; h < SPB; ++h) {
                        const int bs = (CYC == 2 ? (blk & 1) : 0) * SPB + h;
                        const int as = h;  // expert modes: TMEM A stage; router: shared-memory A stage
                        const uint32_t ap = blk & 1;
                        if (!mbar_wait2(&S.full_a[as], ap, &S.full_b[bs], bpar, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < SS; ++j) {
                            const uint32_t blo = b_lo + static_cast<uint32_t>((bs * SS + j) * (kBBytes >> 4));
                            if (dequant_mode) {
                                // A from tensor memory: stage h at 128 h, matrix m at + 64 m,
                                // k-step j at + 32 j (64 K elements = 32 columns)
                                const uint32_t at = ta + static_cast<uint32_t>(h * 128 + j * 32 + mat * 64);
#pragma unroll
                                for (int kk = 0; kk < kBK / 16; ++kk) {
                                    const uint32_t acc = ((kb - kb0) | h | j | kk) != 0;
                                    umma_ts(dm, at + kk * 8, desc64(blo + kk * 2, b_hi), idesc, acc);
                                }
                            } else {
                                const uint32_t alo = a_lo + static_cast<uint32_t>(as * (2 * kABytes >> 4) + mat * (kABytes >> 4));
#pragma unroll
                                for (int kk = 0; kk < kBK / 16; ++kk) {
                                    const uint32_t acc = ((kb - kb0) | h | kk) != 0;
                                    umma_ss(dm, desc64(alo + kk * 2, a_hi), desc64(blo + kk * 2, b_hi), idesc, acc);
                                }
                            }
                        }
                        // expert modes: one release per stage; the dequantisers wait on the
                        // B slot of the same stage one block back
                        if (!dequant_mode) umma_commit(&S.empty_a[as]);
                        umma_commit(&S.empty_b[bs]);
                    }
                }
                if (!ok) break;
                umma_commit(&S.full_acc[ab]);
                if (++ab == n_acc) {
                    ab = 0;
                    acc_ph ^= 1;
                }
            }
            // All tensor-core work of this CTA must finish before TMEM is freed.
            umma_commit(&S.drain);
            drain_wait(&S.drain, 0, status);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------ dequantisers
        if (dequant_mode) {
            const int mi = (warp - 4) >> 2;              // which matrix of the pair
            const int r = ((warp - 4) & 3) * 32 + lane;  // row within the 128-row tile
            const int sw = r & 7;                        // 128-byte swizzle of this row
            const int ngroups = g.K / kBK;
            const bool vec8 = (ngroups & 7) == 0;
            // this warp's TMEM lane quarter holds rows [32 * (warp % 4), +32)
            const uint32_t ta_row = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kTmemAOffset +
                                    static_cast<uint32_t>(mi * 64);
            int blk = 0;
            bool ok = true;
            bool have_pre = false;  // s_nxt / b_nxt already hold the next unit's first register block
            uint4 s_nxt = make_uint4(0u, 0u, 0u, 0u), b_nxt = s_nxt;
            for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
                const Unit u = unit_info<MODE>(g, tile, n_routed);
                if (u.rows <= 0) continue;
                int r0, r1;
                a_rows<MODE>(g, u, r0, r1);
                const int row = (mi ? r1 : r0) + r;
                const uint16_t *srow = (u.shared ? (mi ? g.ss1 : g.ss0) : (mi ? g.s1 : g.s0)) + static_cast<size_t>(row) * ngroups;
                const uint16_t *brow = (u.shared ? (mi ? g.sb1 : g.sb0) : (mi ? g.b1 : g.b0)) + static_cast<size_t>(row) * ngroups;
                // the next unit this CTA runs (tile + gridDim.x, when it has rows)
                const uint16_t *nsrow = nullptr, *nbrow = nullptr;
                {
                    // warm L2 with the next unit's scale / bias rows of this thread
                    const int nt = tile + gridDim.x;
                    if (nt < total_tiles) {
                        const Unit un = unit_info<MODE>(g, nt, n_routed);
                        if (un.rows > 0) {
                            int n0, n1;
                            a_rows<MODE>(g, un, n0, n1);
                            const size_t nrow = static_cast<size_t>((mi ? n1 : n0) + r) * ngroups;
                            nsrow = (un.shared ? (mi ? g.ss1 : g.ss0) : (mi ? g.s1 : g.s0)) + nrow;
                            nbrow = (un.shared ? (mi ? g.sb1 : g.sb0) : (mi ? g.b1 : g.b0)) + nrow;
                            prefetch_l2(nsrow);
                            prefetch_l2(nbrow);
                        }
                    }
                }
                // scale / bias of 8 consecutive groups (two blocks) per 16-byte register
                // block, fetched one register block ahead; groups past K read as zero.
                // In gate/up the refill that would fetch past K fetches the next
                // unit's first register block instead.
                uint4 s_cur, b_cur;
                if (have_pre) {
                    s_cur = s_nxt;
                    b_cur = b_nxt;
                    have_pre = false;
                } else {
                    s_cur = load_groups8(srow, 0, ngroups, vec8);
                    b_cur = load_groups8(brow, 0, ngroups, vec8);
                }
                s_nxt = load_groups8(srow, 8, ngroups, vec8);
                b_nxt = load_groups8(brow, 8, ngroups, vec8);
                for (int kb = 0; kb < KB; ++kb, ++blk) {
                    if ((kb & 1) == 0 && kb > 0) {
                        s_cur = s_nxt;
                        b_cur = b_nxt;
                        const int gn = kb * kBlk + 8;  // first group of the block to fetch
                        if (MODE == kModeGateUp && gn >= ngroups && nsrow) {
                            // this unit needs no further block (kb + 2 >= KB)
                            s_nxt = load_groups8(nsrow, 0, ngroups, vec8);
                            b_nxt = load_groups8(nbrow, 0, ngroups, vec8);
                            have_pre = true;
                        } else {
                            s_nxt = load_groups8(srow, gn, ngroups, vec8);
                            b_nxt = load_groups8(brow, gn, ngroups, vec8);
                        }
                    }
                    const int rs = blk & 1;
                    const uint32_t rpar = (blk >> 1) & 1;
                    // this block's four groups of the 8-group register block
                    const uint2 s_blk = (kb & 1) ? make_uint2(s_cur.z, s_cur.w) : make_uint2(s_cur.x, s_cur.y);
                    const uint2 b_blk = (kb & 1) ? make_uint2(b_cur.z, b_cur.w) : make_uint2(b_cur.x, b_cur.y);
                    const uint8_t *rowp = S.raw[rs][mi] + r * kRawRow;
#pragma unroll
                    for (int h = 0; h < SPB; ++h) {
                        // Each warp runs on its own: lane 0 polls the mbarriers and
                        // broadcasts the result.
                        int go = 0;
                        if (lane == 0) {
                            bool w = ok;
                            if (w && h == 0) w = mbar_wait(&S.full_r[rs], rpar, abort_flag, status);
                            // TMEM A stage h was last read by the MMAs of the same stage one
                            // block back, which released that block's B slot h
                            if (w)
                                w = mbar_wait(&S.empty_b[(CYC == 2 ? ((blk & 1) ^ 1) : 0) * SPB + h],
                                              (CYC == 2 ? ((blk - 1) >> 1) : (blk - 1)) & 1, abort_flag, status);
                            go = w;
                        }
                        const bool got = __shfl_sync(0xffffffffu, go, 0) != 0;
                        if (!got) ok = false;
                        tc_fence_after();  // the MMAs that read this TMEM stage are complete
                        if (got) {
#pragma unroll
                            for (int j = 0; j < SS; ++j) {
                                const int jr = h * SS + j;  // k-step within the block
                                const uint16_t sc = pick16x4(s_blk, jr), bi = pick16x4(b_blk, jr);
                                // 128-byte rows written by TMA with the 128-byte swizzle:
                                // 16-byte chunk c of row r sits at chunk c ^ (r % 8)
                                const uint4 q0 = *reinterpret_cast<const uint4 *>(rowp + (((2 * jr) ^ sw) << 4));
                                const uint4 q1 = *reinterpret_cast<const uint4 *>(rowp + (((2 * jr + 1) ^ sw) << 4));
                                const __half2 b2 = half2_from_bf16_bits(bi);
                                const __half2 s8 = __hmul2(half2_from_bf16_bits(sc), __floats2half2_rn(8.0f, 8.0f));
                                const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                                uint32_t cols[32];  // TMEM column 4c + i holds K positions 8c + 2i, 8c + 2i + 1
#pragma unroll
                                for (int cc = 0; cc < 8; ++cc) {
                                    const uint4 o = dequant8_f16_e2m3(words[cc], s8, b2);
                                    cols[4 * cc + 0] = o.x;
                                    cols[4 * cc + 1] = o.y;
                                    cols[4 * cc + 2] = o.z;
                                    cols[4 * cc + 3] = o.w;
                                }
                                tmem_st_32x32b_x32(ta_row + static_cast<uint32_t>(h * 128 + j * 32), cols);
                            }
                            tmem_st_wait();
                            tc_fence_before();
                        }
                        __syncwarp();
                        if (lane == 0 && ok) {
                            mbar_arrive(&S.full_a[h]);
                            if (h == SPB - 1) mbar_arrive(&S.empty_r[rs]);
                        }
                    }
                }
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------ epilogue (8 warps)
        // Two warps per TMEM lane quarter; they split the accumulator columns in
        // 16-column chunks (even / odd chunks).
        const int ew = warp & 3;             // TMEM lane quarter this warp may access
        const int half = (warp - 12) >> 2;   // which chunks of columns
        const int et = ew * 32 + lane;       // accumulator row (weight row within the tile)
        const int eid = (warp - 12) * 32 + lane;  // 0..255
        int ab = 0;
        uint32_t acc_ph = 0;
        bool ok = true;
        const int n_acc = dequant_mode ? 1 : 2;
        // gate/up: out = 0 for the down projection that follows, this CTA's slice,
        // written a share after each unit (not all at the start, where it would
        // compete with the first units' copies) and the rest at the end
        int64_t zpos = 0, zend = 0, zstep = 0;
        if (MODE == kModeGateUp) {
            const int64_t n4 = static_cast<int64_t>(g.T) * g.d / 4;
            const int64_t per = (n4 + gridDim.x - 1) / gridDim.x;
            zpos = min(n4, blockIdx.x * per);
            zend = min(n4, zpos + per);
            const int my_units = total_tiles > static_cast<int>(blockIdx.x)
                                     ? (total_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                                     : 1;
            zstep = ((zend - zpos + my_units - 1) / my_units + 255) / 256 * 256;
        }
        auto zero_out = [&](int64_t n) {
            float4 *o = reinterpret_cast<float4 *>(g.out);
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            const int64_t stop = min(zend, zpos + n);
            for (int64_t i = zpos + eid; i < stop; i += 256) o[i] = z;
            zpos = stop;
        };
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            int ut, kb0, kb1;
            k_range(tile, ut, kb0, kb1);
            const Unit u = unit_info<MODE>(g, ut, n_routed);
            if (u.rows <= 0) continue;
            if (MODE == kModeDown && eid < u.rows) {
                int tok = u.p0 + eid;
                float wt = 1.0f;
                if (!u.shared) {
                    const int a = g.perm[u.p0 + eid];
                    tok = a / g.top_k;
                    wt = g.topk_w[a];
                }
                if (tok < 0 || tok >= g.T) {
                    record_error(status, kErrDeviceIndex);
                    tok = 0;
                    wt = 0.0f;
                }
                S.ep_tok[eid] = tok;
                S.ep_w[eid] = wt;
            }
            // one thread waits for the accumulator; the group-wide result keeps the
            // warp-collective tcgen05.ld below uniform
            if (eid == 0) {
                bool go = ok;
#ifdef LILY_TEST_STALL_T
                // Test builds only: for T == LILY_TEST_STALL_T the first unit's
                // accumulator wait is preceded by a wait on a barrier that nothing
                // completes, so the bounded wait runs out and the abort path
                // (every role gives up, in-flight copies and MMAs drain, TMEM is
                // freed) executes.
                if (go && g.T == LILY_TEST_STALL_T && tile == static_cast<int>(blockIdx.x))
                    go = mbar_wait(&S.never, 0, abort_flag, status);
#endif
                S.ep_go = go && mbar_wait(&S.full_acc[ab], acc_ph, abort_flag, status);
            }
            named_barrier_sync(kBarEpilogue, 256);  // also publishes ep_tok / ep_w
            const bool got = S.ep_go != 0;
            if (!got) ok = false;
            if (got) {
                tc_fence_after();
                const uint32_t t0 = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(ab * 2 * kTileM);
                const uint32_t t1 = t0 + kTileM;
                if (MODE == kModeGateUp) {
                    // this thread's column chunks c0 = 16 half + 32 q: h = silu(gate) up
                    // packed as fp16 pairs in registers, so the accumulator is released
                    // before the stores
                    uint32_t hp[kTileN / 32][8];
                    bool inf = false;
#pragma unroll
                    for (int q = 0; q < kTileN / 32; ++q) {
                        const int c0 = half * 16 + 32 * q;
                        if (c0 < u.n_mma) {
                            uint32_t v0[16], v1[16];
                            tmem_ld_32x32b_x16(t0 + c0, v0);
                            tmem_ld_32x32b_x16(t1 + c0, v1);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const __half2 hv = __floats2half2_rn(
                                    silu_f(__uint_as_float(v0[2 * j])) * __uint_as_float(v1[2 * j]),
                                    silu_f(__uint_as_float(v0[2 * j + 1])) * __uint_as_float(v1[2 * j + 1]));
                                hp[q][j] = *reinterpret_cast<const uint32_t *>(&hv);
                                // only this unit's tokens count (padding columns hold other rows)
                                const uint32_t a = hp[q][j] & 0x7FFF7FFFu;
                                inf |= (c0 + 2 * j < u.rows && (a & 0xFFFFu) == 0x7C00u) |
                                       (c0 + 2 * j + 1 < u.rows && (a >> 16) == 0x7C00u);
                            }
                        }
                    }
                    if (inf) record_error(status, kErrDeviceRange);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.empty_acc[ab]);
                    // h columns in the K order of dequant8_f16_e2m3 (the down GEMM's A)
                    const int hcol = kperm8_e2m3(u.mt * kTileM + et);
                    const size_t prow0 = u.shared ? static_cast<size_t>(g.T) * g.top_k + u.p0 : static_cast<size_t>(u.p0);
                    __half *hbase = g.h + prow0 * g.I + hcol;
#pragma unroll
                    for (int q = 0; q < kTileN / 32; ++q) {
                        const int c0 = half * 16 + 32 * q;
                        if (c0 < u.n_mma) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int n = c0 + j;
                                if (n < u.rows)
                                    hbase[static_cast<size_t>(n) * g.I] =
                                        __ushort_as_half(static_cast<unsigned short>(hp[q][j >> 1] >> (16 * (j & 1))));
                            }
                        }
                    }
                } else if (MODE == kModeDown) {
                    float *obase = g.out + u.mt * 2 * kTileM + et;
                    for (int c0 = half * 16; c0 < u.n_mma; c0 += 32) {
                        uint32_t v0[16], v1[16];
                        tmem_ld_32x32b_x16(t0 + c0, v0);
                        tmem_ld_32x32b_x16(t1 + c0, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int n = c0 + j;
                            if (n < u.rows) {
                                float *orow = obase + static_cast<size_t>(S.ep_tok[n]) * g.d;
                                const float wt = S.ep_w[n];
                                atomicAdd(orow, wt * __uint_as_float(v0[j]));
                                atomicAdd(orow + kTileM, wt * __uint_as_float(v1[j]));
                            }
                        }
                    }
                } else {
                    // one K split: partial sums without the bias, in the split's slice
                    float bias0 = 0.0f, bias1 = 0.0f;
                    if (g.router_bias && KS == 1) {
                        bias0 = g.router_bias[et];
                        bias1 = g.router_bias[kTileM + et];
                    }
                    float *lbase = (KS == 1 ? g.logits : g.logits_part + static_cast<size_t>(tile - ut * KS) * g.T * g.E) +
                                   static_cast<size_t>(u.p0) * g.E + et;
                    for (int c0 = half * 16; c0 < u.n_mma; c0 += 32) {
                        uint32_t v0[16], v1[16];
                        tmem_ld_32x32b_x16(t0 + c0, v0);
                        tmem_ld_32x32b_x16(t1 + c0, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int n = c0 + j;
                            if (n < u.rows) {
                                float *lrow = lbase + static_cast<size_t>(n) * g.E;
                                lrow[0] = __uint_as_float(v0[j]) + bias0;
                                lrow[kTileM] = __uint_as_float(v1[j]) + bias1;
                            }
                        }
                    }
                }
                if (MODE != kModeGateUp) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.empty_acc[ab]);
                }
            }
            named_barrier_sync(kBarEpilogue, 256);  // ep_tok / ep_w free for the next unit
            if (++ab == n_acc) {
                ab = 0;
                acc_ph ^= 1;
            }
            if (MODE == kModeGateUp) zero_out(zstep);
        }
        if (MODE == kModeGateUp) zero_out(zend - zpos);
    }

    __syncwarp();  // every role reconverges its warp before the CTA-wide barrier
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// Before the expert GEMMs: xs = fp16(x) in routing order with K permuted
// inside each group of 8 (the order the dequantisers write the weights in):
// row p < T top_k is token perm[p] / top_k, row T top_k + t is token t (the
// shared expert's rows).  One warp per token: it reads the token's row of x
// once (8 16-byte loads in flight per lane), converts it once and writes it to
// the token's top_k routed rows inv[t top_k + j] and to its shared row.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_kperm(const uint4 v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
        f[2 * j] = q.x;
        f[2 * j + 1] = q.y;
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // slot pairs (0,2) (4,6) (1,3) (5,7): the order of dequant8_f16_e2m3
        const int e = (j & 1) * 4 + (j >> 1);
        const __half2 hv = __floats2half2_rn(f[e], f[e + 2]);
        o[j] = *reinterpret_cast<const uint32_t *>(&hv);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// WPT warps per token (1, 2, 4 or 8): warp `part` of a token converts every
// WPT-th 32-element stretch of the row, so that few tokens still spread over
// all SMs.
template <int WPT>
__global__ void __launch_bounds__(256) prep_experts_kernel(const uint4 *x, const int *inv, uint4 *xs, int T, int d8,
                                                           int top_k, int *status)
{
    constexpr int wpt = WPT;
    const int lane = threadIdx.x & 31;
    const int64_t routed = static_cast<int64_t>(T) * top_k;
    const int stride = gridDim.x * 8;
    pdl_trigger();
    pdl_wait();  // the inverse permutation is complete
    for (int tw = blockIdx.x * 8 + (threadIdx.x >> 5); tw < T * wpt; tw += stride) {
        const int t = tw / wpt, part = tw - t * wpt;
        // lane j < top_k holds the row of slot j; lane top_k the shared expert's row
        int64_t row = -1;
        if (lane < top_k) {
            const int p = __ldg(inv + static_cast<int64_t>(t) * top_k + lane);
            if (p >= 0 && p < routed)
                row = p;
            else
                record_error(status, kErrDeviceIndex);
        } else if (lane == top_k) {
            row = routed + t;
        }
        const uint4 *src = x + static_cast<int64_t>(t) * d8;
        for (int i0 = part * 32; i0 < d8; i0 += 256 * wpt) {
            uint4 v[8];
            bool inf = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * 32 * wpt + lane;
                if (i < d8) {
                    v[j] = bf16x8_to_f16x8_kperm(__ldg(src + i));
                    inf |= f16x2_has_inf(v[j].x) | f16x2_has_inf(v[j].y) | f16x2_has_inf(v[j].z) |
                           f16x2_has_inf(v[j].w);
                }
            }
            if (inf) record_error(status, kErrDeviceRange);
            for (int k = 0; k <= top_k; ++k) {  // the token's top_k routed rows and its shared row
                const int64_t r = __shfl_sync(0xffffffffu, row, k);
                if (r < 0) continue;
                uint4 *dst = xs + r * d8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = i0 + j * 32 * wpt + lane;
                    if (i < d8) dst[i] = v[j];
                }
            }
        }
    }
}

// inv[perm[p]] = p, for routing tables that come from an earlier call.
__global__ void __launch_bounds__(256) invert_perm_kernel(const int *perm, int *inv, int n, int *status)
{
    pdl_trigger();
    pdl_wait();
    for (int p = blockIdx.x * 256 + threadIdx.x; p < n; p += gridDim.x * 256) {
        const int a = __ldg(perm + p);
        if (a >= 0 && a < n)
            inv[a] = p;
        else
            record_error(status, kErrDeviceIndex);
    }
}

}  // namespace

cudaError_t launch_prep_experts(const uint16_t *x, const int *inv, __half *xs, int T, int d, int top_k, int *status,
                                cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // warps per token: about 16 warps per SM in all, at most 8 per token
    int wpt = 1;
    while (wpt < 8 && static_cast<int64_t>(T) * wpt < static_cast<int64_t>(sms) * 16) wpt *= 2;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((static_cast<int64_t>(T) * wpt + 7) / 8, sms * 8)));
    auto kernel = wpt == 8 ? prep_experts_kernel<8> : wpt == 4 ? prep_experts_kernel<4>
                                                  : wpt == 2 ? prep_experts_kernel<2> : prep_experts_kernel<1>;
    return launch_pdl(kernel, dim3(grid), dim3(256), 0, stream, reinterpret_cast<const uint4 *>(x), inv,
                      reinterpret_cast<uint4 *>(xs), T, d / 8, top_k, status);
}

cudaError_t launch_invert_perm(const int *perm, int *inv, int n, int *status, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    const int grid = std::max(1, std::min((n + 255) / 256, 4096));
    return launch_pdl(invert_perm_kernel, dim3(grid), dim3(256), 0, stream, perm, inv, n, status);
}

size_t grouped_gemm_smem_bytes() { return sizeof(Smem) + 1024; }

template <int MODE>
static cudaError_t launch_mode(const GemmArgs &g, const CUtensorMap &tmB, const CUtensorMap &tmA0, const CUtensorMap &tmA1,
                               const CUtensorMap &tmSA0, const CUtensorMap &tmSA1, int grid, cudaStream_t stream)
{
    const size_t smem = grouped_gemm_smem_bytes();
    const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(grouped_gemm_kernel<MODE>),
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(grouped_gemm_kernel<MODE>, dim3(grid), dim3(kThreads), smem, stream, g, tmB, tmA0, tmA1, tmSA0,
                      tmSA1);
}

cudaError_t launch_grouped_gemm(const GemmArgs &g, const CUtensorMap &tmB, const CUtensorMap &tmA0,
                                const CUtensorMap &tmA1, const CUtensorMap &tmSA0, const CUtensorMap &tmSA1,
                                int grid, cudaStream_t stream)
{
    switch (g.mode) {
    case kModeRouter: return launch_mode<kModeRouter>(g, tmB, tmA0, tmA1, tmSA0, tmSA1, grid, stream);
    case kModeGateUp: return launch_mode<kModeGateUp>(g, tmB, tmA0, tmA1, tmSA0, tmSA1, grid, stream);
    case kModeDown: return launch_mode<kModeDown>(g, tmB, tmA0, tmA1, tmSA0, tmSA1, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace lily
