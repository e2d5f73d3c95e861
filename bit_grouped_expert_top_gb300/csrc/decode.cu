// Decode path of the MoE layer for 1..8 tokens: one persistent kernel runs the
// whole chain of layers.
//
// Method (page "Perplexity libera o Lily", noticiai.com.br, section "Prefill e
// decode: onde estao os ganhos"): at batch 1 there is almost no weight reuse,
// so memory bandwidth sets the ceiling.  Only the bytes of the selected experts
// (plus the shared expert and the router) are read, each exactly once, with
// coalesced bulk copies, dequantised in registers (weights rounded once to
// fp16, as in the prefill path) and multiplied with fp32 accumulation.  The
// page's decode step overlaps its kernels by tracking the real dependencies
// between them; here those dependencies are carried by data inside one
// resident kernel instead of kernel boundaries.
//
// GB300 design.  One CTA per SM (a cooperative launch, so every CTA is
// resident), 8 compute warps and 1 producer warp.  Per layer l, every CTA:
//   A  builds the layer input x_l in shared memory (layer 0: x; later layers:
//      bf16 of the previous output over sqrt(mean(out^2) + 1e-6), the
//      parameter-free RMS norm that links layers), reading the previous
//      layer's output words from the exchange area;
//   -  computes its one or two router rows (logit of expert c and c + G) and
//      publishes them;
//   B  reads all 256 x T logits, selects the top 8 per token (lower index first
//      among equal logits) and builds the list of distinct experts ("units":
//      the shared expert is unit 0 with weight 1); computes its shared-expert
//      gate/up rows (if any) while the routed experts' bytes load;
//   -  gate/up tasks (unit, 8 rows of I): tensor-core GEMV (mma.sync m16n8k16,
//      the tokens as the 8 columns, gate rows and up rows as the two 8-row
//      halves of the tile), SwiGLU in registers, scaled by the unit's routing
//      weight, published as fp16 h';
//   C  down tasks (16 output rows): the sum over all units of Wd_u h'_u in one
//      fragment (deterministic), published as the layer output.
// Data moves between CTAs through workspace buffers (double buffered by layer
// parity) and per-layer ready counters: a writer stores its part, then one
// thread adds 1 to the counter with release semantics; one thread of each
// reading CTA polls that one counter with acquire loads until every writer has
// signalled, and the CTA then reads the data from L2.  No grid-wide barrier is
// involved, and the polling touches one word per CTA (polling the data itself,
// with every CTA spinning on the same lines, queued up at the L2 slices).  The
// counters are per layer and zeroed at the start of every call.
//
// Every weight a CTA needs streams through a ring of shared-memory slots.  A
// producer warp copies the weight rows of each item with bulk (TMA) copies
// (2 KB to 8 KB each) and the 256-512 byte scale/bias slices as 16-byte
// cp.async pieces from its 32 lanes; the compute warps release a slot after
// reading it.  (One SM's TMA unit takes 30-50 ns to start each bulk copy
// whatever its size, so the small slices, four per gate/up task and two per
// down unit, go through the load/store units instead; and with the compute
// warps issuing cp.async themselves they stalled on the full load queue
// instead of working on the items already there.)
// Items that do not depend on the routing (the router rows and the shared
// expert's gate/up rows) of layer l + 1 are issued as soon as the slots of
// layer l free up, so they load while layer l finishes; the routed experts'
// gate/up rows and then the down rows of all units are issued the moment the
// top-8 is known.
//
// Every wait (mbarrier or ready counter) is bounded; a wait that runs out
// records LILY_ERR_DEVICE_TIMEOUT, raises a global abort flag that the other
// CTAs see, and every CTA leaves its layer loop at the next top-8 point and
// waits for its own copies in flight before it exits.
#include <algorithm>

#include "lily_device.cuh"
#include "lily_internal.h"

namespace lily {
namespace {

constexpr int kMaxT = kDecodeMaxT;
constexpr int kMaxUnits = kDecodeMaxUnits;
constexpr int kCW = 8;                        // compute warps
constexpr int kDecThreads = (kCW + 1) * 32;   // + the producer warp
constexpr int kProdWarp = kCW;
constexpr int kComputeThreads = kCW * 32;
constexpr int kKB = 128;                      // K block of one lane pass (16 bytes of int4 per row)
constexpr int kGURows = 8;                    // I rows of one gate/up task
constexpr int kDownRows = 16;                 // output rows of one down task
constexpr int kMaxSlots = 16;
constexpr int kSmemLimit = 232448;            // 227 KB of dynamic shared memory per CTA
constexpr int kBarTop8 = 1, kBarCompute = 2;  // named barriers (0 is __syncthreads)

struct DecSmem {
    uint64_t full[kMaxSlots], empty[kMaxSlots];  // ring slot landed / free again
    int abort;                    // this CTA gives up (set by any failed wait)
    int decide;                   // the abort decision taken at the top-8 point
    int n_units;
    int unit_e[kMaxUnits];        // expert of unit u (-1: shared)
    float unit_w[kMaxUnits][kMaxT];
    int umask[256];               // tokens that selected expert e (bit n)
    int sel_e[kMaxT][8];          // the top-8 of each token and their weights
    float sel_w[kMaxT][8];
    int scan_tmp[kCW];
    float inv_rms[kMaxT];
    float rred[kCW][2][kMaxT];
    float sred[kCW][kMaxT];
    uint2 zeros[8];
    float red[2][kCW][32][4];     // cross-warp sums of mma fragments, double buffered
};

__host__ __device__ constexpr size_t align128(size_t v) { return (v + 127) / 128 * 128; }
constexpr size_t kStaticBytes = align128(sizeof(DecSmem));

// Bytes of one ring slot: a gate/up task (8 rows of gate and up, K = d, with
// scales and biases) = 9d, or one unit of a down task (16 rows, K = I) = 9I.
__host__ __device__ inline size_t slot_bytes_of(int d, int I)
{
    return align128(static_cast<size_t>(9) * (d > I ? d : I));
}
// Staged h' of one down item: units per item (slot / 9I) x I/128 K blocks x T
// tokens x 64 payload words of 4 bytes.
__host__ __device__ inline size_t stage_bytes(int T, int d, int I)
{
    const size_t upc = slot_bytes_of(d, I) / (static_cast<size_t>(9) * I);
    return align128(upc * (I / 128) * T * 64 * 4);
}

// ---------------------------------------------------------------- memory helpers

// Bulk (TMA) copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Ready counters: release add by the writer, acquire load by the reader.
__device__ __forceinline__ void signal_ready(unsigned int *p)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_flag(const int *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_flag(int *p, int v)
{
    asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Waiter {
    volatile int *s_abort;
    int *g_abort;
    int *status;
};

__device__ __forceinline__ void raise_abort(const Waiter &w)
{
    *w.s_abort = 1;
    st_flag(w.g_abort, 1);
}

// Waits (one thread) until the counter reaches `target`; bounded, gives up on
// an abort raised in this CTA or by another one.
__device__ __forceinline__ bool wait_ready(const unsigned int *p, unsigned int target, const Waiter &w)
{
    uint64_t t0 = 0;
#pragma unroll 1
    for (int iter = 0;; ++iter) {
        if (ld_acquire(p) >= target) return true;
        if (*w.s_abort) return false;
        if ((iter & 15) == 15 && ld_flag(w.g_abort)) {
            *w.s_abort = 1;
            return false;
        }
        const uint64_t now = global_timer_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > LILY_WAIT_LIMIT_NS) {
            record_error(w.status, kErrDeviceTimeout);
            raise_abort(w);
            return false;
        }
    }
}

// mbarrier wait (bounded; a failure also raises the global abort flag).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const Waiter &w)
{
    if (mbar_wait(bar, parity, w.s_abort, w.status)) return true;
    raise_abort(w);
    return false;
}

__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

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

__device__ __forceinline__ void compute_sync() { named_barrier_sync(kBarCompute, kComputeThreads); }

// ---------------------------------------------------------------- tensor-core GEMV
// The expert GEMVs run on mma.sync m16n8k16 (f16 x f16 -> f32): 16 weight rows
// x 16 K x 8 token columns per instruction (tokens >= T are zero columns), so a
// weight is dequantised once for all tokens.  Lane (g = lane / 4, t = lane % 4)
// reads 16 bytes (32 weights) of rows g and g + 8 for each 128-wide K block:
// weights [32 t, 32 t + 32) of the block.  The K order inside the block is
// permuted so that these weights are exactly this lane's A-fragment entries:
// within 32-bit word w (weights 8w..8w+7, rebuilt in pairs (0,2) (4,6) (1,3)
// (5,7) by dequant8_f16_e2m3), weight e goes to slice 2w + (e & 1), entry
// e >> 1 of the lane's four K positions.  The B operand (x, or h' for the down
// projection) is stored in the same permuted order, so each lane reads its B
// fragment of a slice as one 8-byte value: layout [K block][token][t][slice][4].
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 128-wide K block of a 16-row tile: q_g / q_g8 hold this lane's 16 bytes of
// rows g and g + 8, sb_g / sb_g8 the bf16 scale (low half) and bias (high
// half) of its group; b holds the lane's B fragments of the block (8 slices).
__device__ __forceinline__ void mma_kblock(float (&d)[4], uint4 q_g, uint4 q_g8, uint32_t sb_g, uint32_t sb_g8,
                                           const uint2 (&b)[8])
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
        const uint32_t a0[4] = {pg.x, pg8.x, pg.y, pg8.y};  // slice 2w: pairs (0,2) and (4,6)
        const uint32_t a1[4] = {pg.z, pg8.z, pg.w, pg8.w};  // slice 2w + 1: pairs (1,3) and (5,7)
        mma_16816(d, a0, b[2 * w].x, b[2 * w].y);
        mma_16816(d, a1, b[2 * w + 1].x, b[2 * w + 1].y);
    }
}

// Scale and bias of group `grp` of row `row`, packed (scale low, bias high).
__device__ __forceinline__ uint32_t sb_of(const uint16_t *s, const uint16_t *b, int row, int ngroups, int grp)
{
    return static_cast<uint32_t>(s[row * ngroups + grp]) | (static_cast<uint32_t>(b[row * ngroups + grp]) << 16);
}

// Eight bf16 inputs (k0..k0+7 of one token) -> fp16 in the permuted B order
// (x0 x2 x4 x6 | x1 x3 x5 x7); raises the range flag on an infinite result.
__device__ __forceinline__ uint4 bf16x8_to_perm_f16(uint4 v, bool &inf)
{
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
    const uint4 o = make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                               *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
    inf |= f16x2_has_inf(o.x) | f16x2_has_inf(o.y) | f16x2_has_inf(o.z) | f16x2_has_inf(o.w);
    return o;
}

// Half offset of K element k0 (a multiple of 8) of token n in the permuted B
// layout [k / 128][T][4][8][4].
__device__ __forceinline__ int perm_b_offset(int k0, int n, int T)
{
    const int kb = k0 >> 7, r = k0 & 127, t4 = r >> 5, w = (r >> 3) & 3;
    return (((kb * T + n) * 4 + t4) * 8 + 2 * w) * 4;
}

// ---------------------------------------------------------------- per-CTA work plan
// Gate/up tasks j = 0 .. U * I/8 - 1 (unit j / (I/8), I rows 8 (j % (I/8)) ..),
// task j on CTA G - 1 - (j mod G); down tasks (16 output rows) k = c, c + G.
struct Plan {
    int G, c, nu_gu;       // CTAs, this CTA, gate/up tasks per unit (I / 8)
    int n_down, n_mydown;  // down tasks in all, of this CTA (0..2)
    int upc;               // units per down item
    int n_rrows;           // router rows of this CTA (1 or 2)
    __device__ int gu_first() const { return G - 1 - c; }
};

template <typename F>
__device__ __forceinline__ void for_gu_tasks(const Plan &p, int j_lo, int j_hi, F &&f)
{
    for (int j = p.gu_first(); j < j_hi; j += p.G)
        if (j >= j_lo) f(j);
}

// ---------------------------------------------------------------- the kernel
// 9 warps: one SM sub-partition holds 3 of them, so at most 168 registers each
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a)
{
    extern __shared__ __align__(128) uint8_t dsm[];
    DecSmem &S = *reinterpret_cast<DecSmem *>(dsm);
    const int T = a.T, d = a.d, I = a.I, E = a.E;
    __nv_bfloat16 *xb = reinterpret_cast<__nv_bfloat16 *>(dsm + kStaticBytes);     // [T][d] bf16
    __half *xp = reinterpret_cast<__half *>(dsm + kStaticBytes + static_cast<size_t>(T) * d * 2);  // permuted fp16
    // h' of one down item's units, staged from the exchange buffer: [unit][K block][T][4][16] words
    uint32_t *hs = reinterpret_cast<uint32_t *>(dsm + kStaticBytes + align128(static_cast<size_t>(T) * d * 4));
    uint8_t *ring = dsm + kStaticBytes + align128(static_cast<size_t>(T) * d * 4) + stage_bytes(T, d, I);
    const int tid = threadIdx.x;  // compute threads 0..255, producer warp 256..287
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int NS = a.n_slots;
    const uint32_t SB = static_cast<uint32_t>(a.slot_bytes);
    const Waiter wt{&S.abort, a.abort_flag, &a.ctrl->status};

    Plan P;
    P.G = gridDim.x;
    P.c = blockIdx.x;
    P.nu_gu = I / kGURows;
    P.n_down = d / kDownRows;
    P.n_mydown = (P.c < P.n_down) + (P.c + P.G < P.n_down);
    P.upc = static_cast<int>(SB / (9u * I));
    P.n_rrows = (P.c < E) + (P.c + P.G < E);
    const int nkb_d = d / kKB, nkb_i = I / kKB;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&S.full[s], 33);     // the bulk copies' byte count, then the producer's 32 lanes
            mbar_init(&S.empty[s], kCW);   // the compute warps, each once done reading
        }
        S.abort = 0;
        S.decide = 0;
        S.unit_e[0] = -1;  // unit 0 is always the shared expert
        fence_mbar_init();
    }
    if (tid < 8) S.zeros[tid] = make_uint2(0u, 0u);
    __syncthreads();

    // Abort decision at the top-8 point of every layer, the same for all warps:
    // one thread reads the flag between two barriers of the whole CTA.  The
    // producer learns here that the unit list of the layer is complete.
    auto top8_point = [&]() -> bool {
        named_barrier_sync(kBarTop8, kDecThreads);
        if (tid == 0) S.decide = *reinterpret_cast<volatile int *>(&S.abort);
        named_barrier_sync(kBarTop8, kDecThreads);
        return *reinterpret_cast<volatile int *>(&S.decide) != 0;
    };

    // ---------------------------------------------------------------- the ring
    // Items, in the order they are issued and consumed, per layer li:
    //   router rows of this CTA; the shared expert's gate/up tasks of this CTA;
    //   [top-8 point]  the routed gate/up tasks of this CTA; per down task,
    //   chunks of units [u0, u0 + upc).
    // The producer warp copies the weight rows of an item with bulk (TMA)
    // copies, counted in bytes on the slot's full barrier, and the small
    // scale/bias slices with 16-byte cp.async pieces spread over its 32 lanes,
    // each lane arriving (noinc) once its pieces land; the barrier fires when
    // both are complete.  Only the producer waits on the copy engines; the
    // compute warps work on the items already there.  Item n goes to slot n % NS once its previous
    // occupant has been released by all compute warps.
    if (warp == kProdWarp) {
        uint32_t pit = 0;  // items issued
        bool pok = true;
        auto copy_seg = [&](uint8_t *dst, const void *src, uint32_t bytes) {
            for (uint32_t o = static_cast<uint32_t>(lane) * 16u; o < bytes; o += 32u * 16u)
                cp_async_16(dst + o, static_cast<const uint8_t *>(src) + o);
        };
        // waits for a free slot and announces the item's bulk-copy bytes;
        // returns the slot, or -1 when giving up
        auto begin_item = [&](uint32_t bulk_bytes) -> int {
            if (!pok) return -1;
            const int slot = static_cast<int>(pit % NS);
            int ok = 1;
            if (lane == 0) {
                ok = wait_bar(&S.empty[slot], ((pit / NS) & 1) ^ 1, wt);
                if (ok) mbar_arrive_expect_tx(&S.full[slot], bulk_bytes);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) pok = false;
            return ok ? slot : -1;
        };
        auto end_item = [&](int slot) {
            cp_async_mbar_arrive_noinc(&S.full[slot]);
            ++pit;
        };
        // gate/up task j of expert e (e < 0: the shared expert)
        auto issue_gu = [&](const DecodeLayerPtrs &W, int j, int e) {
            const int slot = begin_item(8u * d);
            if (slot < 0) return;
            uint8_t *base = ring + static_cast<size_t>(slot) * SB;
            const size_t r0 = (e < 0 ? 0 : static_cast<size_t>(e) * I) + static_cast<size_t>(j % P.nu_gu) * kGURows;
            const size_t ng = d / 64;
            // rows: two bulk copies; scale/bias slices: cp.async pieces
            if (lane == 0) bulk_g2s(base, (e < 0 ? W.sh_gate_q : W.gate_q) + r0 * (d / 2), 4u * d, &S.full[slot]);
            if (lane == 1) bulk_g2s(base + 4 * d, (e < 0 ? W.sh_up_q : W.up_q) + r0 * (d / 2), 4u * d, &S.full[slot]);
            copy_seg(base + 8 * d, (e < 0 ? W.sh_gate_s : W.gate_s) + r0 * ng, d / 4);
            copy_seg(base + 8 * d + d / 4, (e < 0 ? W.sh_gate_b : W.gate_b) + r0 * ng, d / 4);
            copy_seg(base + 8 * d + d / 2, (e < 0 ? W.sh_up_s : W.up_s) + r0 * ng, d / 4);
            copy_seg(base + 8 * d + 3 * d / 4, (e < 0 ? W.sh_up_b : W.up_b) + r0 * ng, d / 4);
            end_item(slot);
        };
        // units [u0, u1) of down task k: 16 rows of Wd of each unit's expert
        auto issue_down = [&](const DecodeLayerPtrs &W, int k, int u0, int u1) {
            const int slot = begin_item(8u * I * (u1 - u0));
            if (slot < 0) return;
            uint8_t *base = ring + static_cast<size_t>(slot) * SB;
            const size_t j0 = static_cast<size_t>(P.c + k * P.G) * kDownRows;
            const size_t ng = I / 64;
            for (int i = 0; i < u1 - u0; ++i) {
                const int e = S.unit_e[u0 + i];
                const size_t r0 = (e < 0 ? 0 : static_cast<size_t>(e) * d) + j0;
                uint8_t *ub = base + static_cast<size_t>(i) * 9 * I;
                if (lane == i) bulk_g2s(ub, (e < 0 ? W.sh_down_q : W.down_q) + r0 * (I / 2), 8u * I, &S.full[slot]);
                copy_seg(ub + 8 * I, (e < 0 ? W.sh_down_s : W.down_s) + r0 * ng, I / 2);
                copy_seg(ub + 8 * I + I / 2, (e < 0 ? W.sh_down_b : W.down_b) + r0 * ng, I / 2);
            }
            end_item(slot);
        };
        for (int li = 0; li < a.n_layers; ++li) {
            const DecodeLayerPtrs &W = a.L[li];
            {
                const int slot = begin_item(2u * d * P.n_rrows);
                if (slot >= 0) {
                    uint8_t *base = ring + static_cast<size_t>(slot) * SB;
                    if (lane < P.n_rrows)
                        bulk_g2s(base + static_cast<size_t>(lane) * 2 * d,
                                 W.router_w + static_cast<size_t>(P.c + lane * P.G) * d, 2u * d, &S.full[slot]);
                    end_item(slot);
                }
            }
            for_gu_tasks(P, 0, P.nu_gu, [&](int j) { issue_gu(W, j, -1); });
            if (top8_point()) break;
            const int U = S.n_units;
            for_gu_tasks(P, P.nu_gu, U * P.nu_gu, [&](int j) { issue_gu(W, j, S.unit_e[j / P.nu_gu]); });
            for (int k = 0; k < P.n_mydown; ++k)
                for (int u0 = 0; u0 < U; u0 += P.upc) issue_down(W, k, u0, min(U, u0 + P.upc));
        }
        // no copy into this CTA's shared memory may still be in flight at exit
        cp_async_wait_all();
        return;
    }

    uint32_t cit = 0;  // index of the next item to consume
    int rp = 0;        // red buffer parity
    const size_t TD = static_cast<size_t>(T) * d;
    const size_t HX = static_cast<size_t>(kMaxUnits) * nkb_i * T * 64;  // words of one h' buffer
    auto ready_of = [&](int l) { return a.ready + static_cast<size_t>(l) * kDecodeReadySlots; };

    // Waits for the next item; returns its slot base (nullptr: giving up).  The
    // result is uniform within each warp.
    auto take_item = [&](int &slot_out) -> const uint8_t * {
        const int slot = static_cast<int>(cit % NS);
        const bool got = wait_bar(&S.full[slot], (cit / NS) & 1, wt);
        ++cit;
        slot_out = slot;
        return __all_sync(0xffffffffu, got) ? ring + static_cast<size_t>(slot) * SB : nullptr;
    };
    // This warp is done reading the item's slot.  An item whose copies did not
    // arrive (giving up) is not released: the slot may still be written.
    auto release_item = [&](int slot, const uint8_t *base) {
        __syncwarp();
        if (lane == 0 && base) mbar_arrive(&S.empty[slot]);
    };

    // ---- layer input x_l into xb (bf16) and xp (permuted fp16); export_only:
    // only write x_next[l - 1] (the normalised output of the last layer)
    auto build_input = [&](int l, bool export_only) {
        bool inf = false;
        if (l == 0) {
            for (int q = tid; q < T * (d / 8); q += kComputeThreads) {
                const int n = q / (d / 8), k0 = (q - n * (d / 8)) * 8;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.x_in + static_cast<size_t>(n) * d + k0));
                *reinterpret_cast<uint4 *>(xb + static_cast<size_t>(n) * d + k0) = v;
                *reinterpret_cast<uint4 *>(xp + perm_b_offset(k0, n, T)) = bf16x8_to_perm_f16(v, inf);
            }
        } else {
            const float *src = a.out_x + static_cast<size_t>((l - 1) & 1) * TD;
            if (tid == 0) wait_ready(ready_of(l - 1) + 1, static_cast<unsigned int>(P.n_down), wt);
            compute_sync();
#pragma unroll
            for (int n = 0; n < kMaxT; ++n) {
                if (n < T) {
                    float ss = 0.0f;
                    for (int k0 = tid * 8; k0 < d; k0 += kComputeThreads * 8) {
                        const float4 *p = reinterpret_cast<const float4 *>(src + static_cast<size_t>(n) * d + k0);
                        const float4 v0 = __ldcg(p), v1 = __ldcg(p + 1);
                        ss = fmaf(v0.x, v0.x, fmaf(v0.y, v0.y, fmaf(v0.z, v0.z, fmaf(v0.w, v0.w, ss))));
                        ss = fmaf(v1.x, v1.x, fmaf(v1.y, v1.y, fmaf(v1.z, v1.z, fmaf(v1.w, v1.w, ss))));
                    }
                    ss = warp_sum(ss);
                    if (lane == 0) S.sred[warp][n] = ss;
                }
            }
            compute_sync();
            if (tid < T) {
                float s = 0.0f;
                for (int w = 0; w < kCW; ++w) s += S.sred[w][tid];
                S.inv_rms[tid] = 1.0f / sqrtf(s / static_cast<float>(d) + 1e-6f);
            }
            compute_sync();
            for (int q = tid; q < T * (d / 8); q += kComputeThreads) {
                const int n = q / (d / 8), k0 = (q - n * (d / 8)) * 8;
                const float r = S.inv_rms[n];
                const float4 *p = reinterpret_cast<const float4 *>(src + static_cast<size_t>(n) * d + k0);
                const float4 v0 = __ldcg(p), v1 = __ldcg(p + 1);
                const __nv_bfloat162 b0 = __floats2bfloat162_rn(v0.x * r, v0.y * r), b1 = __floats2bfloat162_rn(v0.z * r, v0.w * r);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(v1.x * r, v1.y * r), b3 = __floats2bfloat162_rn(v1.z * r, v1.w * r);
                const uint4 v = make_uint4(*reinterpret_cast<const uint32_t *>(&b0), *reinterpret_cast<const uint32_t *>(&b1),
                                           *reinterpret_cast<const uint32_t *>(&b2), *reinterpret_cast<const uint32_t *>(&b3));
                if (blockIdx.x == 0 && a.x_next)
                    *reinterpret_cast<uint4 *>(a.x_next + static_cast<size_t>(l - 1) * TD + static_cast<size_t>(n) * d + k0) = v;
                if (!export_only) {
                    *reinterpret_cast<uint4 *>(xb + static_cast<size_t>(n) * d + k0) = v;
                    *reinterpret_cast<uint4 *>(xp + perm_b_offset(k0, n, T)) = bf16x8_to_perm_f16(v, inf);
                }
            }
        }
        if (inf) record_error(wt.status, kErrDeviceRange);
        compute_sync();
    };

    // ---- gate/up task j of unit u: h' = w_u silu(gate x) (up x), published
    auto gu_task = [&](int l, int j, int u) {
        int slot;
        const uint8_t *base = take_item(slot);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (base) {
            const uint8_t *gq = base, *uq = base + 4 * d;
            const uint16_t *gs = reinterpret_cast<const uint16_t *>(base + 8 * d);
            const uint16_t *gb = reinterpret_cast<const uint16_t *>(base + 8 * d + d / 4);
            const uint16_t *us = reinterpret_cast<const uint16_t *>(base + 8 * d + d / 2);
            const uint16_t *ub = reinterpret_cast<const uint16_t *>(base + 8 * d + 3 * d / 4);
            const int ng = d / 64;
            for (int kb = warp; kb < nkb_d; kb += kCW) {
                const uint4 qg = lds128(gq + g * (d / 2) + kb * 64 + t * 16);
                const uint4 qu = lds128(uq + g * (d / 2) + kb * 64 + t * 16);
                const int grp = 2 * kb + (t >> 1);
                uint2 bfr[8];
                const uint2 *src = g < T ? reinterpret_cast<const uint2 *>(xp + (((kb * T + g) * 4 + t) * 8) * 4) : S.zeros;
#pragma unroll
                for (int s = 0; s < 8; ++s) bfr[s] = src[s];
                mma_kblock(acc, qg, qu, sb_of(gs, gb, g, ng, grp), sb_of(us, ub, g, ng, grp), bfr);
            }
        }
        release_item(slot, base);
        float *r = S.red[rp][warp][lane];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = acc[q];
        compute_sync();
        if (warp == 0 && base != nullptr) {
            float D[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = 0; w < kCW; ++w)
#pragma unroll
                for (int q = 0; q < 4; ++q) D[q] += S.red[rp][w][lane][q];
            // D[0], D[1]: gate row g, tokens 2t, 2t+1; D[2], D[3]: up row g
            uint32_t hh[2];
            bool inf = false;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int n = 2 * t + m;
                const float wu = n < T ? S.unit_w[u][n] : 0.0f;
                const __half h = __float2half_rn(wu * silu_f(D[m]) * D[2 + m]);
                inf |= __hisinf(h);
                hh[m] = __half_as_ushort(h);
            }
            if (inf) record_error(wt.status, kErrDeviceRange);
            // pair row g with row g + 2 (lane + 8): the two halves of one word
            const uint32_t ph0 = __shfl_down_sync(0xffffffffu, hh[0], 8);
            const uint32_t ph1 = __shfl_down_sync(0xffffffffu, hh[1], 8);
            if ((g & 2) == 0) {
                const int i0 = (j % P.nu_gu) * kGURows;
                const int kbI = i0 >> 7, r0 = i0 & 127, t4 = r0 >> 5, w8 = (r0 >> 3) & 3;
                const int s = 2 * w8 + (g & 1), pw = g >> 2;
                uint32_t *hx = a.h_x + static_cast<size_t>(l & 1) * HX;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int n = 2 * t + m;
                    if (n < T) {
                        const size_t idx = ((((static_cast<size_t>(u) * nkb_i + kbI) * T + n) * 4 + t4) * 8 + s) * 2 + pw;
                        hx[idx] = hh[m] | ((m ? ph1 : ph0) << 16);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) signal_ready(ready_of(l) + 2 + u);
        }
        rp ^= 1;
    };

    // ---- down item: units [u0, u1) of one down task, accumulated into acc.
    // Once the item's units are ready, all compute threads copy its h' words
    // into `hs`, then each warp runs its (unit, K block) pairs.
    auto down_item = [&](int l, int u0, int u1, float(&acc)[4]) {
        int slot;
        const uint8_t *base = take_item(slot);
        const int nw = (u1 - u0) * nkb_i * T * 64;  // words of the item
        const uint32_t *hx = a.h_x + static_cast<size_t>(l & 1) * HX + static_cast<size_t>(u0) * nkb_i * T * 64;
        if (tid == 0)
            for (int u = u0; u < u1; ++u) wait_ready(ready_of(l) + 2 + u, static_cast<unsigned int>(P.nu_gu), wt);
        compute_sync();
        for (int w0 = tid * 4; w0 < nw; w0 += kComputeThreads * 4)
            *reinterpret_cast<uint4 *>(hs + w0) = __ldcg(reinterpret_cast<const uint4 *>(hx + w0));
        compute_sync();
        if (base) {
            const int ng = I / 64;
            for (int pi = warp; pi < (u1 - u0) * nkb_i; pi += kCW) {
                const int i = pi / nkb_i, kb = pi - i * nkb_i;
                const uint8_t *ubase = base + static_cast<size_t>(i) * 9 * I;
                const uint16_t *s = reinterpret_cast<const uint16_t *>(ubase + 8 * I);
                const uint16_t *b = reinterpret_cast<const uint16_t *>(ubase + 8 * I + I / 2);
                uint2 bfr[8];
                const uint2 *src =
                    g < T ? reinterpret_cast<const uint2 *>(hs + ((static_cast<size_t>(pi) * T + g) * 4 + t) * 16) : S.zeros;
#pragma unroll
                for (int q = 0; q < 8; ++q) bfr[q] = src[q];
                const uint4 qg = lds128(ubase + g * (I / 2) + kb * 64 + t * 16);
                const uint4 qg8 = lds128(ubase + (g + 8) * (I / 2) + kb * 64 + t * 16);
                const int grp = 2 * kb + (t >> 1);
                mma_kblock(acc, qg, qg8, sb_of(s, b, g, ng, grp), sb_of(s, b, g + 8, ng, grp), bfr);
            }
        }
        release_item(slot, base);
        compute_sync();  // hs is reused by the next item
    };

    // ---- down task k done: sum the warps' fragments, publish the rows
    auto finish_down = [&](int l, int k, float(&acc)[4]) {
        float *r = S.red[rp][warp][lane];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = acc[q];
        compute_sync();
        if (warp == 0) {
            float D[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = 0; w < kCW; ++w)
#pragma unroll
                for (int q = 0; q < 4; ++q) D[q] += S.red[rp][w][lane][q];
            const int j0 = (P.c + k * P.G) * kDownRows;
            float *ox = a.out_x + static_cast<size_t>(l & 1) * TD;
            float *out = a.out + static_cast<size_t>(l) * TD;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = 2 * t + (q & 1), j = j0 + g + 8 * (q >> 1);
                if (n < T) {
                    out[static_cast<size_t>(n) * d + j] = D[q];
                    ox[static_cast<size_t>(n) * d + j] = D[q];
                }
            }
            __syncwarp();
            if (lane == 0) signal_ready(ready_of(l) + 1);
        }
        rp ^= 1;
    };

    for (int li = 0; li < a.n_layers; ++li) {
        const int l = a.layer0 + li;
        const DecodeLayerPtrs &W = a.L[li];

        // ---- A: input, router rows
        build_input(l, false);
        {
            int slot;
            const uint8_t *base = take_item(slot);
            float part[2][kMaxT];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int n = 0; n < kMaxT; ++n) part[r][n] = 0.0f;
            if (base) {
                const int kw = d / kCW;
                for (int k0 = warp * kw + lane * 8; k0 < (warp + 1) * kw; k0 += 256) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        if (r < P.n_rrows) {
                            const uint4 wv = lds128(base + static_cast<size_t>(r) * 2 * d + k0 * 2);
#pragma unroll
                            for (int n = 0; n < kMaxT; ++n)
                                if (n < T) part[r][n] = dot8_bf16(wv, lds128(xb + static_cast<size_t>(n) * d + k0), part[r][n]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int n = 0; n < kMaxT; ++n)
                    if (r < P.n_rrows && n < T) {
                        const float v = warp_sum(part[r][n]);
                        if (lane == 0) S.rred[warp][r][n] = v;
                    }
            release_item(slot, base);
            compute_sync();
            if (warp == 0) {
                if (tid < P.n_rrows * T && base) {
                    const int r = tid / T, n = tid - r * T, e = P.c + r * P.G;
                    float v = 0.0f;
                    for (int w = 0; w < kCW; ++w) v += S.rred[w][r][n];
                    if (W.router_bias) v += W.router_bias[e];
                    a.logits_x[(static_cast<size_t>(l & 1) * T + n) * E + e] = v;
                    if (a.trace_logits) a.trace_logits[(static_cast<size_t>(l) * T + n) * E + e] = v;
                }
                __syncwarp();
#ifdef LILY_TEST_STALL_DECODE_LAYERS
                // Test builds only: in a call of exactly this many layers, CTA 0
                // never signals its logits of layer 3, so every CTA's bounded wait
                // for them runs out and the abort path executes.
                if (!(a.last_launch && a.layer0 + a.n_layers == LILY_TEST_STALL_DECODE_LAYERS && l == 3 &&
                      blockIdx.x == 0))
#endif
                    if (lane == 0) signal_ready(ready_of(l));
            }
        }
        // ---- B: top-8 per token and the unit list
        if (tid < kMaxT) S.unit_w[0][tid] = 1.0f;  // unit 0: the shared expert, weight 1
        S.umask[tid] = 0;
        if (tid == 0) wait_ready(ready_of(l), static_cast<unsigned int>(P.G), wt);
        compute_sync();
        if (warp < T) {
            {
                const float4 *p = reinterpret_cast<const float4 *>(a.logits_x + (static_cast<size_t>(l & 1) * T + warp) * E + lane * 8);
                const float4 l0 = __ldcg(p), l1 = __ldcg(p + 1);
                const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                int sel_e;
                float sel_w;
                warp_top8_keys(lv, lane, sel_e, sel_w);
                if (lane < 8) {
                    if (blockIdx.x == 0 && a.trace_idx) a.trace_idx[(static_cast<size_t>(l) * T + warp) * 8 + lane] = sel_e;
                    if (blockIdx.x == 0 && a.trace_w) a.trace_w[(static_cast<size_t>(l) * T + warp) * 8 + lane] = sel_w;
                    atomicOr(&S.umask[sel_e], 1 << warp);
                    S.sel_e[warp][lane] = sel_e;
                    S.sel_w[warp][lane] = sel_w;
                }
            }
        }
        compute_sync();
        {
            const int used = S.umask[tid] != 0;
            int incl = used;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += nb;
            }
            if (lane == 31) S.scan_tmp[warp] = incl;
            compute_sync();
            int off = 0, n_used = 0;
            for (int w = 0; w < kCW; ++w) {
                if (w < warp) off += S.scan_tmp[w];
                n_used += S.scan_tmp[w];
            }
            if (used) {
                const int u = 1 + off + incl - used;
                S.unit_e[u] = tid;
                const int m = S.umask[tid];
#pragma unroll
                for (int n = 0; n < kMaxT; ++n) {
                    float wv = 0.0f;
                    if ((m >> n) & 1)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (S.sel_e[n][j] == tid) wv = S.sel_w[n][j];
                    S.unit_w[u][n] = wv;
                }
            }
            if (tid == 0) S.n_units = min(n_used + 1, kMaxUnits);
        }
        if (top8_point()) break;  // the producer issues the routed experts' bytes from here
        const int U = S.n_units;

        // ---- the shared expert's gate/up rows of this CTA (computed while the
        // routed experts' bytes, issued at the top-8 point, are in flight)
        for_gu_tasks(P, 0, P.nu_gu, [&](int j) { gu_task(l, j, 0); });

        // ---- C: routed gate/up, then per down task the down rows of every unit
        for_gu_tasks(P, P.nu_gu, U * P.nu_gu, [&](int j) { gu_task(l, j, j / P.nu_gu); });
        for (int k = 0; k < P.n_mydown; ++k) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int u0 = 0; u0 < U; u0 += P.upc) down_item(l, u0, min(U, u0 + P.upc), acc);
            finish_down(l, k, acc);
        }
    }
    // the normalised output of the last layer (the input a next layer would take)
    if (a.last_launch && a.x_next && blockIdx.x == 0 && !*reinterpret_cast<volatile int *>(&S.decide))
        build_input(a.layer0 + a.n_layers, true);
}

}  // namespace

int decode_slot_bytes(int d, int I) { return static_cast<int>(slot_bytes_of(d, I)); }

size_t decode_smem_bytes(int T, int d, int I, int n_slots)
{
    return kStaticBytes + align128(static_cast<size_t>(T) * d * 4) + stage_bytes(T, d, I) +
           static_cast<size_t>(n_slots) * decode_slot_bytes(d, I);
}

int decode_ring_slots(int T, int d, int I)
{
    const size_t fixed = decode_smem_bytes(T, d, I, 0);
    if (fixed >= static_cast<size_t>(kSmemLimit)) return 0;
    const int n = static_cast<int>(std::min<size_t>(kMaxSlots, (kSmemLimit - fixed) / decode_slot_bytes(d, I)));
    return n >= 3 ? n : 0;
}

// Ring slots of a launch on the current device: at most decode_ring_slots(),
// fewer if the device cannot keep one CTA with that much shared memory
// resident on every SM (a cooperative launch needs every CTA resident).
int decode_launch_slots(int T, int d, int I)
{
    for (int n = decode_ring_slots(T, d, I); n >= 3; --n) {
        const int smem = static_cast<int>(decode_smem_bytes(T, d, I, n));
        if (set_max_dynamic_smem(reinterpret_cast<const void *>(decode_kernel), smem) != cudaSuccess) continue;
        int blocks = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, decode_kernel, kDecThreads, smem) == cudaSuccess &&
            blocks >= 1)
            return n;
    }
    return 0;
}

cudaError_t launch_decode(const DecodeArgs &a, int grid, cudaStream_t stream)
{
    const size_t smem = decode_smem_bytes(a.T, a.d, a.I, a.n_slots);
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(decode_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // cooperative: every CTA is resident at once (CTAs wait on each other's data)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel, a);
}

}  // namespace lily
