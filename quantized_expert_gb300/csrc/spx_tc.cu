// spx_tc.cu -- verify experts on the fifth-generation tensor cores: tcgen05
// products with accumulators in tensor memory, operands staged by TMA tensor
// copies; the layer call takes this path for verify calls of 9 tokens or more.
//
// [P1 Key Contributions 4: expert-wise verification reordering turns the
// per-token expert GEMVs into one dense product per expert over the tokens it
// holds.]  The expert launch (spx_engine.cu) keeps every activation row of the
// call in shared memory and issues mma.sync tiles of 8 tokens, so its weight
// ring shrinks as the token count grows and above ~24 tokens (4096-wide: ~17)
// its geometry runs out.  This path streams activation tiles next to the
// weight tiles, so its shared memory does not grow with the token count, and
// one thread issues the products, leaving the other warps to the epilogue:
//
//   gather launch   x rows of each active expert (and every token for the
//                   shared expert) copied into one block of rows per expert
//                   slot; the shared-expert gate per token; the slots' ready
//                   counts zeroed.
//   product launch  gate/up units, then down units:
//                   gate/up unit = (slot, 64 columns of I): D[128 x Np] =
//                   A . B^T with A = 64 gate rows and 64 up rows of the expert
//                   ([I][H], k = H), B = the slot's Np token rows; epilogue
//                   h = silu(gate) * up (fp16) into the slot's h rows, then
//                   the slot's ready count;
//                   down unit = (slot, 128 rows of H, a piece of I): D[128 x
//                   Np] = Wd . h^T, read once the slot's ready count is full;
//                   epilogue: each token's share, scaled by its routing weight
//                   (or the shared gate), added to the fp32 accumulator of its
//                   output row.
//   output launch   out = fp16(accumulator); the accumulator is cleared.
//
// Every launch is a programmatic dependent of the one before it.
//
// Weights come in this path's own pack (spx_f16_tc_repack): per expert, the
// gate/up tiles (unit u, k-chunk kc) and then the down tiles (128-row block
// hb, k-chunk kc), each tile 128 rows x 64 fp16 = 16 KB contiguous, so one
// 3-D tensor copy streams a whole tile from consecutive addresses (the
// canonical [I][H] rows would be 128 pieces of 128 B, 4-8 KB apart) and the
// TMA unit applies the shared-memory swizzle.  Gate/up tile row 32q + i is
// gate column 64u + 16q + i (i < 16) or up column 64u + 16q + i - 16.
//
// Inside a block (one per SM, persistent over units): warp 0 lane 0 issues
// the TMA copies into a 9-stage ring (A 16 KB + B up to 8 KB per stage, k =
// 64 per stage, 128-byte swizzle), warp 1 lane 0 issues tcgen05.mma (M = 128,
// N = Np = tokens rounded up to 16, K = 16 per instruction, fp16 inputs, fp32
// accumulate) into one of two tensor-memory accumulators, and warps 2-5 drain
// the other accumulator with tcgen05.ld (warp w reads lanes 32*(w%4)..+31).
// Every wait is bounded: a wait that runs out records SPX_ERR_TIMEOUT (site
// SITE_TC) and the block leaves its loops, waits for its own copies and
// products in flight (bounded too), frees its tensor memory and returns.
#include <cuda.h>  // CUtensorMap and the tensor-map encoder's argument types
#include <string.h>

#include "spx_internal.cuh"

namespace spx {

namespace {

constexpr int kTcStages = 9;
constexpr int kTcKc = 64;                           // k per stage: one 128-byte swizzled row
constexpr int kTcABytes = 128 * kTcKc * 2;          // 16 KB: 128 rows
constexpr int kTcBMaxBytes = kMaxT * kTcKc * 2;     // 8 KB: up to 64 token rows
constexpr int kTcStageBytes = kTcABytes + kTcBMaxBytes;
constexpr int kTcThreads = 192;                     // producer, issuer, 4 epilogue warps
constexpr uint32_t kTcAccCols = 64;                 // columns of one accumulator (Np <= 64)
constexpr uint32_t kTcTmemCols = 2 * kTcAccCols;    // two accumulators, a power of two >= 32
constexpr int kTcSlotBytes = 2 * (kMaxE + 1) * 4;    // expert and token count per slot
static_assert((kMaxE + 1) * 4 <= 3072, "the ready counts fit between the gate and the rows of the scratch");
constexpr size_t kTcSmem = 1024 + (size_t)kTcStages * kTcStageBytes + 256 + kTcSlotBytes;
static_assert(kMaxT <= 64, "one accumulator holds every token of a slot");

struct TcParams {
    CUtensorMap tm_w, tm_sw;  // routed / shared packs: [tiles][128 rows][64]
    CUtensorMap tm_xs, tm_hs; // [nslot*npm][H], [nslot*npm][Imax]
    const __half *x;
    const __half *w_sgate;
    const int32_t *active, *n_active;
    const TokTable *tables;
    __half *xs, *hs;
    float *gam, *acc;
    uint32_t *ready;  // per slot: epilogue warps done with a gate/up unit of the slot (4 per unit)
    __half *out;
    WsHeader *hdr;
    uint64_t budget;
    int T, H, E, I, I_s, npm, Imax, has_shared;
    int nslot;  // 1 + min(E, T*k)
};
static_assert(sizeof(TcParams) <= sizeof(TcPlan) && alignof(TcParams) <= alignof(TcPlan), "a plan holds the params");

// ------------------------------------------------------------- PTX ----
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *tm, int x, int y, int z, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// D (tensor memory) (+)= A (shared, descriptor) . B (shared, descriptor)^T
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every product this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 32 lanes (this warp's quarter) x 16 consecutive 32-bit columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by a TMA copy with
// 128-byte swizzle: rows of 128 B (64 fp16 of k), 8-row groups 1024 B apart.
// Fields: start address >> 4 (bits 0-13), leading offset (16-29, unused for
// swizzled K-major tiles), stride offset 1024 >> 4 (32-45), descriptor
// version 1 (46-47), base offset 0 (49-51: the tile starts on a 1024-byte
// boundary), swizzle mode 2 = 128 B (61-63).  The k-th group of 16 columns of
// a row starts 32*k bytes further (the swizzle is applied to the final
// address).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort, const TcParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > p.budget) {
            record_timeout(&p.hdr->status, SITE_TC);
            *abort = 1;
            return false;
        }
    }
}
// Drain wait after an abort: ignores the abort flag, gives up after `ns`.
__device__ __forceinline__ void tc_drain(uint64_t *bar, uint32_t parity, uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < ns) {
    }
}

__device__ __forceinline__ int tc_nact(const TcParams &p) {
    const int na = *p.n_active;
    return na < 0 ? 0 : (na > p.E ? p.E : na);
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// One unit of work, decoded the same way by every role of a block.
struct TcUnit {
    bool down; // a down unit (else gate/up)
    int slot;  // 0 = shared expert, 1 + a = active expert a
    int e;     // expert id (routed) or -1
    int n;     // tokens of the slot
    int pos;   // gate/up: first column of I; down: first row of H
    int kc0;   // first k stage (a down unit covers one piece of its k range)
    int nk;    // k stages
};

// gate/up units: the shared expert's I_s/64 first, then every active expert's I/64
__device__ __forceinline__ int tc_gu_count(const TcParams &p, int nact) {
    return (p.has_shared ? p.I_s / kTcKc : 0) + nact * (p.I / kTcKc);
}
// Down units cut their k range (I or I_s) into pieces of at most
// min(I, H)/64/m stages, as equal as possible: no unit is longer than a
// gate/up unit; the pieces' partial sums meet in the accumulator.  m (1..3) is
// chosen per launch from the unit count: the one that minimises rounds over
// the grid x (stages per piece + kTcUnitCost), so that the last round of units
// stays short.  kTcUnitCost, a unit's fixed cost in stages, was bracketed on
// GB300: the DeepSeek-shaped layer at 17 tokens (624 units of 22 stages, 4.1
// rounds, or 1248 of 11) ran faster with m = 1, so it exceeds 2.75; the
// Phi-shaped one (832 units of 50 stages or 1664 of 25) faster with m = 2, so
// it is below 5.  Every block computes the same m from n_active.
constexpr int kTcUnitCost = 4;
struct TcSplit {
    int pieces, len;  // pieces per 128-row block, k stages per piece (the last may be shorter)
};
__device__ __forceinline__ TcSplit tc_split(const TcParams &p, int ks, int m) {
    const int lim = max(1, min(p.I, p.H) / kTcKc / m);  // I and H are multiples of 64
    TcSplit d;
    d.pieces = ks > 0 ? (ks + lim - 1) / lim : 0;
    d.len = ks > 0 ? (ks + d.pieces - 1) / d.pieces : 0;
    return d;
}
// down units: the shared expert's (H/128 blocks x pieces) first, then every active expert's
__device__ __forceinline__ int tc_dn_count_m(const TcParams &p, int nact, int m) {
    const int sh = p.has_shared ? (p.H / 128) * tc_split(p, p.I_s / kTcKc, m).pieces : 0;
    return sh + nact * (p.H / 128) * tc_split(p, p.I / kTcKc, m).pieces;
}
__device__ __forceinline__ int tc_down_m(const TcParams &p, int nact, int grid) {
    int best = 1;
    long long best_cost = -1;
    for (int m = 1; m <= 3; ++m) {
        const int len = tc_split(p, p.I / kTcKc, m).len;
        const long long cost = (long long)((tc_dn_count_m(p, nact, m) + grid - 1) / grid) * (len + kTcUnitCost);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = m;
        }
    }
    return best;
}
// slot_e / slot_n: expert and token count of every slot, staged in shared
// memory once per block (slot 0, the shared expert: -1 and T).  A unit with
// t.n == 0 or t.nk == 0 is skipped by every role alike.
// Units of the product launch: the ngu gate/up units, then the down units.
__device__ __forceinline__ TcUnit tc_unit(const TcParams &p, int u, const int *slot_e, const int *slot_n, int m,
                                          int ngu) {
    TcUnit t;
    t.down = u >= ngu;
    if (!t.down) {
        const int ns = p.has_shared ? p.I_s / kTcKc : 0;
        const int per = p.I / kTcKc;
        int a = -1, v = u;
        if (u >= ns) {
            a = (u - ns) / per;
            v = u - ns - a * per;
        }
        t.slot = 1 + a;
        t.e = a < 0 ? -1 : slot_e[1 + a];
        t.n = a < 0 ? p.T : slot_n[1 + a];
        t.pos = kTcKc * v;
        t.kc0 = 0;
        t.nk = p.H / kTcKc;
        return t;
    }
    u -= ngu;
    const TcSplit ds = tc_split(p, p.I_s / kTcKc, m), dr = tc_split(p, p.I / kTcKc, m);
    const int ns = p.has_shared ? (p.H / 128) * ds.pieces : 0;
    int a = -1, v = u;
    if (u >= ns) {
        const int per = (p.H / 128) * dr.pieces;
        a = (u - ns) / per;
        v = u - ns - a * per;
    }
    const TcSplit d = a < 0 ? ds : dr;
    const int ks = (a < 0 ? p.I_s : p.I) / kTcKc;
    const int hb = v / d.pieces, pc = v - hb * d.pieces;
    t.slot = 1 + a;
    t.e = a < 0 ? -1 : slot_e[1 + a];
    t.n = a < 0 ? p.T : slot_n[1 + a];
    t.pos = 128 * hb;
    t.kc0 = pc * d.len;
    t.nk = max(0, min(d.len, ks - t.kc0));
    return t;
}

// ------------------------------------------------------ gather launch --
// One warp per (slot, row) with slot < 1 + min(E, T*k) and row < T, then one
// warp per token for the shared-expert gate.  Only a slot's n real rows are
// written: the rows up to its 16-row tile hold whatever the workspace held, as
// a token row of the product only ever reaches that token's own output column,
// which the epilogues leave out.
__global__ void __launch_bounds__(256) tc_gather_kernel(const __grid_constant__ TcParams p, int nslot) {
    griddep_launch_dependents();
    griddep_wait();
    const int gtid = (int)(blockIdx.x * blockDim.x + threadIdx.x);
    const int warp = gtid >> 5, lane = threadIdx.x & 31;
    const int nact = tc_nact(p);
    if (gtid < nslot) p.ready[gtid] = 0u;  // the product launch reads them after this launch completes
    if (warp < nslot * p.T) {
        const int slot = warp / p.T, r = warp - slot * p.T;
        if (slot > nact || (slot == 0 && !p.has_shared)) return;
        int tok = r;
        if (slot > 0) {
            int e = p.active[slot - 1];
            e = (e < 0 || e >= p.E) ? 0 : e;
            int n = p.tables[e].n;
            n = (n < 0 || n > p.T) ? 0 : n;
            if (r >= n) return;
            tok = p.tables[e].e[r].tok;
            tok = (tok < 0 || tok >= p.T) ? 0 : tok;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.H);
        uint4 *dst = reinterpret_cast<uint4 *>(p.xs + ((size_t)slot * p.npm + r) * p.H);
        for (int c = lane; c < p.H / 8; c += 32) dst[c] = __ldg(src + c);
        return;
    }
    // shared-expert gate per token: gamma = 1 / (1 + exp(-x . w_sgate)), else 1
    const int t = warp - nslot * p.T;
    if (t >= p.T) return;
    float g = 1.0f;
    if (p.w_sgate) {
        float z = 0.f;
        for (int hh = lane * 2; hh < p.H; hh += 64) {
            const float2 xv = __half22float2(*reinterpret_cast<const __half2 *>(p.x + (size_t)t * p.H + hh));
            const float2 wv = __half22float2(*reinterpret_cast<const __half2 *>(p.w_sgate + hh));
            z = fmaf(xv.x, wv.x, z);
            z = fmaf(xv.y, wv.y, z);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        g = 1.0f / (1.0f + expf(-z));
    }
    if (lane == 0) p.gam[t] = g;
}

// ------------------------------------------------- product launch ------
__device__ __forceinline__ uint32_t tc_ld_acquire(const uint32_t *c) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    return v;
}
// Bounded wait until *c >= target (another block's gate/up epilogues), then
// the h rows they stored may be read by TMA copies (async proxy).
__device__ __forceinline__ bool tc_wait_count(const uint32_t *c, uint32_t target, volatile int *abort,
                                              const TcParams &p) {
    if (tc_ld_acquire(c) < target) {
        const uint64_t t0 = global_timer_ns();
        while (tc_ld_acquire(c) < target) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > p.budget) {
                record_timeout(&p.hdr->status, SITE_TC);
                *abort = 1;
                return false;
            }
            __nanosleep(128);
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Gate/up units of every slot, then the down units, in one persistent launch:
// a down unit's h rows are read once the slot's gate/up units have all been
// drained (its ready count).  Every block takes its gate/up units before any
// down unit, and a block's own epilogue never waits for its producer, so each
// wait ends once the gate/up units ahead of it are done.
__global__ void __launch_bounds__(kTcThreads, 1) tc_mlp_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t tc_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)kTcStages * kTcStageBytes);
    uint64_t *empty = full + kTcStages;
    uint64_t *accf = empty + kTcStages;  // accumulator b holds a finished unit
    uint64_t *acce = accf + 2;           // accumulator b has been read out
    uint64_t *fin = acce + 2;            // products drained (abort path)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *slot_e = reinterpret_cast<int *>(ring + (size_t)kTcStages * kTcStageBytes + 256);
    int *slot_n = slot_e + kMaxE + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tm_w);
        prefetch_tmap(&p.tm_xs);
        prefetch_tmap(&p.tm_hs);
        if (p.has_shared) prefetch_tmap(&p.tm_sw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    griddep_wait();  // routing, token tables, gathered rows and zeroed ready counts are complete
    const int nact = tc_nact(p);
    const int dm = tc_down_m(p, nact, (int)gridDim.x);  // down k-piece multiplier
    const int ngu = tc_gu_count(p, nact);
    const int nunits = ngu + tc_dn_count_m(p, nact, dm);
    for (int a = threadIdx.x; a <= nact; a += blockDim.x) {
        int e = -1, n = p.T;
        if (a > 0) {
            e = p.active[a - 1];
            e = (e < 0 || e >= p.E) ? 0 : e;
            n = p.tables[e].n;
            n = (n < 0 || n > p.T) ? 0 : n;
        }
        slot_e[a] = e;
        slot_n[a] = n;
    }
    __syncthreads();

    if (warp == 0 && lane == 0) {
        // ---- producer: TMA copies of A (weights) and B (token rows) per stage
        const uint64_t pol_w = policy_evict_first(), pol_act = policy_evict_last();
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
            const TcUnit t = tc_unit(p, u, slot_e, slot_n, dm, ngu);
            if (t.n == 0 || t.nk == 0) continue;
            const int nb = (t.n + 15) >> 4;
            const uint32_t bytes = (uint32_t)kTcABytes + (uint32_t)nb * 16 * kTcKc * 2;
            const int brow = t.slot * p.npm;
            for (int kc = 0; kc < t.nk; ++kc, ++it) {
                const int s = (int)(it % kTcStages);
                if (!tc_wait(&empty[s], ((it / kTcStages) & 1) ^ 1, abort_flag, p)) {
                    ok = false;
                    break;
                }
                const int Iw = t.slot == 0 ? p.I_s : p.I;
                // a down unit's h rows: once every gate/up unit of the slot has been drained
                if (t.down && kc == 0 &&
                    !tc_wait_count(p.ready + t.slot, 4u * (uint32_t)(Iw / kTcKc), abort_flag, p)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], bytes);
                uint8_t *sa = ring + (size_t)s * kTcStageBytes, *sb = sa + kTcABytes;
                const int k0 = (t.kc0 + kc) * kTcKc;
                // the unit's tile for this k-chunk (pack order: expert, gate/up tiles, down tiles)
                const int gu_tiles = (Iw / kTcKc) * (p.H / kTcKc);
                const int tile = (t.slot == 0 ? 0 : t.e * (3 * gu_tiles / 2)) +
                                 (t.down ? gu_tiles + (t.pos / 128) * (Iw / kTcKc) : (t.pos / kTcKc) * (p.H / kTcKc)) +
                                 t.kc0 + kc;
                tma_load_3d(sa, t.slot == 0 ? &p.tm_sw : &p.tm_w, 0, 0, tile, &full[s], pol_w);
                const CUtensorMap *tb = t.down ? &p.tm_hs : &p.tm_xs;
                for (int j = 0; j < nb; ++j) tma_load_2d(sb + j * 2048, tb, k0, brow + 16 * j, &full[s], pol_act);
            }
        }
        if (!ok) {
            // copies issued and not yet waited for by the issuer: let them land
            const uint32_t lo = it > (uint32_t)kTcStages ? it - kTcStages : 0u;
            for (uint32_t j = lo; j < it; ++j) tc_drain(&full[j % kTcStages], (j / kTcStages) & 1, 100000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- issuer: tcgen05.mma per stage, commit frees the stage
        uint32_t it = 0, uc = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
            const TcUnit t = tc_unit(p, u, slot_e, slot_n, dm, ngu);
            if (t.n == 0 || t.nk == 0) continue;
            const int b = (int)(uc & 1);
            if (!tc_wait(&acce[b], ((uc >> 1) & 1) ^ 1, abort_flag, p)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)b * kTcAccCols;
            const uint32_t idesc = idesc_f16_f32(128, (t.n + 15) & ~15);
            for (int kc = 0; kc < t.nk; ++kc, ++it) {
                const int s = (int)(it % kTcStages);
                if (!tc_wait(&full[s], (it / kTcStages) & 1, abort_flag, p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(ring + (size_t)s * kTcStageBytes), sb = sa + kTcABytes;
#pragma unroll
                for (int j = 0; j < kTcKc / 16; ++j)
                    umma_f16(d, sw128_desc(sa + 32 * j), sw128_desc(sb + 32 * j), idesc, (kc | j) != 0);
                umma_commit(&empty[s]);
            }
            if (!ok) break;
            umma_commit(&accf[b]);
            ++uc;
        }
        if (*abort_flag) {
            umma_commit(fin);  // everything issued so far has completed once fin flips
            tc_drain(fin, 0, 100000000ull);
        }
    } else if (warp >= 2) {
        // ---- epilogue: drain an accumulator while the other one fills
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        uint32_t uc = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const TcUnit t = tc_unit(p, u, slot_e, slot_n, dm, ngu);
            if (t.n == 0 || t.nk == 0) continue;
            const int b = (int)(uc & 1);
            if (!tc_wait(&accf[b], (uc >> 1) & 1, abort_flag, p)) break;
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)b * kTcAccCols;
            const int np = (t.n + 15) & ~15;
            if (!t.down) {
                // lane l < 16: gate column pos+16q+l; lane l+16: the same up column
                const int col = t.pos + 16 * q + (lane & 15);
                __half *hrow = p.hs + (size_t)t.slot * p.npm * p.Imax + col;
                for (int j = 0; j < np; j += 16) {
                    uint32_t r[16];
                    tmem_ld16(base + (uint32_t)j, r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float mine = __uint_as_float(r[i]);
                        const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
                        if (lane < 16) {
                            const float h = mine / (1.0f + expf(-mine)) * other;
                            hrow[(size_t)(j + i) * p.Imax] = __float2half_rn(h);
                        }
                    }
                }
                __threadfence();  // this lane's h stores, before the slot's ready count
                __syncwarp();
                if (lane == 0) atomicAdd(p.ready + t.slot, 1u);
            } else {
                const int hcol = t.pos + 32 * q + lane;  // output column of this lane
                const TokEntry *ent = t.slot == 0 ? nullptr : p.tables[t.e].e;
                for (int j = 0; j < np; j += 16) {
                    uint32_t r[16];
                    tmem_ld16(base + (uint32_t)j, r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = j + i;
                        if (n < t.n) {
                            int row;
                            float sc;
                            if (ent) {
                                row = ent[n].row;
                                sc = ent[n].scale;
                            } else {
                                row = n;
                                sc = p.gam[n];
                            }
                            row = (row < 0 || row >= p.T) ? 0 : row;
                            atomicAdd(p.acc + (size_t)row * p.H + hcol, sc * __uint_as_float(r[i]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
            ++uc;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

// ------------------------------------------------------ output launch --
__global__ void __launch_bounds__(256) tc_out_kernel(const __grid_constant__ TcParams p) {
    griddep_launch_dependents();
    griddep_wait();
    const int n4 = p.T * p.H / 4;
    float4 *acc4 = reinterpret_cast<float4 *>(p.acc);
    uint2 *out2 = reinterpret_cast<uint2 *>(p.out);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
        const float4 v = __ldcg(acc4 + i);
        uint2 o;
        o.x = h2_as_u32(__floats2half2_rn(v.x, v.y));
        o.y = h2_as_u32(__floats2half2_rn(v.z, v.w));
        out2[i] = o;
        __stcg(acc4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
    }
}

// ------------------------------------------------------------- host ----
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A pack of 16 KB tiles [ntiles][128][64] fp16, copied one whole tile per box
// with 128-byte swizzle.
bool map_tiles(CUtensorMap *m, const void *base, uint64_t ntiles) {
    const EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kTcKc, 128, ntiles};
    const cuuint64_t strides[2] = {(cuuint64_t)kTcKc * 2, (cuuint64_t)kTcABytes};
    const cuuint32_t box[3] = {(cuuint32_t)kTcKc, 128, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 matrix [rows][cols] (row-major, cols % 64 == 0), copied as boxes of 64
// columns x box_rows rows with 128-byte swizzle.
bool map_rows(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    const EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcKc, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaLaunchConfig_t tc_config(dim3 grid, int threads, size_t smem, cudaStream_t s, bool pdl,
                             cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

}  // namespace

// ------------------------------------------------------------ repack --
// One thread per 16-byte piece of the pack: piece p = (tile, row, 8-column
// group) = (p >> 10, (p >> 3) & 127, p & 7).
__global__ void __launch_bounds__(256) tc_repack_kernel(const __half *wg, const __half *wu, const __half *wd, int E,
                                                        int H, int I, uint4 *dst) {
    const int kh = H / kTcKc, ki = I / kTcKc;
    const long long gu = (long long)ki * kh, tpe = gu + (long long)(H / 128) * ki;
    const long long n = (long long)E * tpe * 1024;
    for (long long pc = (long long)blockIdx.x * blockDim.x + threadIdx.x; pc < n;
         pc += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(pc & 7), r = (int)((pc >> 3) & 127);
        const long long t = pc >> 10;
        const int e = (int)(t / tpe);
        long long tt = t - (long long)e * tpe;
        const __half *src;
        if (tt < gu) {
            const int u = (int)(tt / kh), kc = (int)(tt - (long long)u * kh);
            const int q = r >> 5, i = r & 31;
            const int col = kTcKc * u + 16 * q + (i & 15);
            src = (i < 16 ? wg : wu) + ((size_t)e * I + col) * H + kTcKc * kc + 8 * j;
        } else {
            tt -= gu;
            const int hb = (int)(tt / ki), kc = (int)(tt - (long long)hb * ki);
            src = wd + ((size_t)e * H + 128 * hb + r) * I + kTcKc * kc + 8 * j;
        }
        dst[pc] = __ldg(reinterpret_cast<const uint4 *>(src));
    }
}

size_t tc_tiles(int H, int I) { return (size_t)(I / kTcKc) * (H / kTcKc) + (size_t)(H / 128) * (I / kTcKc); }

int launch_tc_repack(const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int E, int H, int I, void *dst,
                     cudaStream_t s) {
    const long long pieces = (long long)E * (long long)tc_tiles(H, I) * 1024;
    const long long blocks = (pieces + 255) / 256;
    tc_repack_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), 256, 0, s>>>(
        reinterpret_cast<const __half *>(wg), reinterpret_cast<const __half *>(wu),
        reinterpret_cast<const __half *>(wd), E, H, I, static_cast<uint4 *>(dst));
    return record_launch(cudaGetLastError());
}

size_t tc_scratch_bytes(int T, int H, int I, int E, int k, int I_s) {
    const size_t nslot = (size_t)(E < T * k ? E : T * k) + 1;
    const size_t npm = (size_t)((T + 15) & ~15);
    const size_t imax = (size_t)(I > I_s ? I : I_s);
    return 4096 + nslot * npm * ((size_t)H + imax) * 2;  // gate, ready counts, rows, h
}

int tc_preload() {
    const int sm = (int)kTcSmem;
    if (cudaFuncSetAttribute(tc_mlp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm) != cudaSuccess)
        return SPX_ERR_CUDA;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, tc_gather_kernel) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, tc_out_kernel) != cudaSuccess)
        return SPX_ERR_CUDA;
    return encode_fn() ? SPX_OK : SPX_ERR_UNSUPPORTED;
}

int tc_plan(const TcArgs &a, TcPlan *plan) {
    static thread_local int loaded_dev = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPX_ERR_CUDA;
    if (loaded_dev != dev) {
        const int st = tc_preload();
        if (st) return st;
        loaded_dev = dev;
    }
    TcParams p;
    memset(&p, 0, sizeof(p));
    const int T = a.T, H = a.H, E = a.E, I = a.I, I_s = a.shared_tc ? a.I_s : 0;
    const int nslot = (E < T * a.k ? E : T * a.k) + 1;
    const int npm = (T + 15) & ~15;
    const int imax = I > I_s ? I : I_s;
    uint8_t *scr = static_cast<uint8_t *>(a.scratch);
    p.gam = reinterpret_cast<float *>(scr);
    p.ready = reinterpret_cast<uint32_t *>(scr + 1024);
    p.xs = reinterpret_cast<__half *>(scr + 4096);
    p.hs = p.xs + (size_t)nslot * npm * H;
    bool ok = map_tiles(&p.tm_w, a.routed_tc, (uint64_t)E * tc_tiles(H, I)) &&
              map_rows(&p.tm_xs, p.xs, H, (uint64_t)nslot * npm, 16) &&
              map_rows(&p.tm_hs, p.hs, imax, (uint64_t)nslot * npm, 16);
    if (ok && I_s) ok = map_tiles(&p.tm_sw, a.shared_tc, tc_tiles(H, I_s));
    if (!ok) return SPX_ERR_UNSUPPORTED;
    p.x = a.x;
    p.w_sgate = I_s ? a.w_sgate : nullptr;
    p.active = a.active;
    p.n_active = a.n_active;
    p.tables = a.tables;
    p.acc = a.acc;
    p.out = a.out;
    p.hdr = a.hdr;
    p.budget = a.wait_budget_ns;
    p.T = T;
    p.H = H;
    p.E = E;
    p.I = I;
    p.I_s = I_s;
    p.npm = npm;
    p.Imax = imax;
    p.has_shared = I_s > 0;
    p.nslot = nslot;
    memcpy(plan->bytes, &p, sizeof(p));
    return SPX_OK;
}

int launch_tc_plan(const TcPlan &plan, cudaStream_t s, bool pdl) {
    const TcParams &p = *reinterpret_cast<const TcParams *>(plan.bytes);
    const int nsm = device_sm_count();
    cudaLaunchAttribute attr[1];
    const int gwarps = (p.nslot + 1) * p.T;  // slot rows, then the gate's tokens
    cudaLaunchConfig_t cfg = tc_config(dim3((gwarps + 7) / 8), 256, 0, s, pdl, attr);
    int st = record_launch(cudaLaunchKernelEx(&cfg, tc_gather_kernel, p, p.nslot));
    if (st) return st;
    cfg = tc_config(dim3(nsm), kTcThreads, kTcSmem, s, true, attr);
    st = record_launch(cudaLaunchKernelEx(&cfg, tc_mlp_kernel, p));
    if (st) return st;
    cfg = tc_config(dim3(4 * nsm), 256, 0, s, true, attr);
    return record_launch(cudaLaunchKernelEx(&cfg, tc_out_kernel, p));
}

}  // namespace spx
