// spx_draft.cu -- the fused multi-expert INT4 draft launch (T <= 5 tokens).
//
// Method (ai.info summary of the Specter paper, Key Contributions 2 and 4;
// richland.au post, "What shipped"): a draft step runs every selected INT4
// (GPTQ, group 128) expert of a layer, plus the FP16 shared expert, in one
// launch, dequantising the INT4 weights while multiplying them with fp16
// activations; the expert MLP is SwiGLU, y = W_d (silu(W_g x) * (W_u x)).
//
// GB300 design.  At T = 1 a layer is ~60-90 MB of weights read once, ~10 us at
// HBM speed, so balance and latency decide everything.  The work is cut into
// ~16 KB items, each processed by ONE consumer warp, with no block barrier:
//   SG  shared gate/up   (16-column block, range of H)
//   RG  routed gate/up   (S-column slice of an active expert, range of H)
//   SD  shared down      (pair of output m-tiles = 32 outputs, range of I_s)
//   RD  routed down      (32 outputs of an active expert, range of I)
// All gate/up items of one column block run on the SM that dequeued the
// block: their partial sums meet in a shared-memory slot, and the warp that
// completes the block applies SiLU, writes the fp16 intermediate h (mma
// B-fragment order) to global memory and counts the block as ready.  So a
// gate/up item costs no global atomics and no fence; only a block's last item
// publishes.  Down items follow every gate/up block in one dynamic queue; their
// weights stream at once, and a poller warp bulk-copies each down item's h
// slice next to them as soon as that slice is complete, so each output gets
// ~2 partial sums per expert, not one per slice.  The producer warp dequeues
// whole blocks (or pairs of down items) with the next ticket already in
// flight, and never waits on h.  Consumer warps take ring stages in order
// through a shared-memory ticket, so a slow item never stalls the others.
// Every block routes the launch's tokens itself (softmax, top-k, the token
// tables of the active experts) in shared memory; block 0 also writes the
// routing outputs.  The launch may begin while the previous one on the stream
// finishes: a block's first queue unit is static, so the producer issues its
// weight copies before it waits for that launch; everything else waits.
#include "spx_internal.cuh"
#include "spx_routing.cuh"
#include "spx_draft_gguf.cuh"
#include "spx_timeline.cuh"

#include <math.h>

#include <atomic>

namespace spx {

enum : int { DK_SG = 0, DK_RG = 1, DK_SD = 2, DK_RD = 3, DK_DONE = 4, DK_NOP = 5 };
// dynamic shared memory of the launch at most (the profiling build keeps its
// marks in static shared memory next to it)
constexpr int kDkSmemLimit = kSmemLimit - (TL_ON ? 4096 : 0);
constexpr int kDkData = 16896;    // largest item: 4 INT4 groups of 32 columns (or 8 of 16)
constexpr int kDkRdGroups = 7;    // INT4 down groups (of 128 rows of I) per RD item
// zero points of an RD item (32 per group) after its largest weight run
constexpr int kDkRdZeroOff = kDkRdGroups * kW4ColGroupBytes;
static_assert(kDkRdZeroOff % 16 == 0 && kDkRdZeroOff + kDkRdGroups * 64 <= kDkData, "RD zero points fit the stage");
// GGUF Q8_0 experts: groups of 128 rows of 4352 bytes, three per routed item
constexpr int kDkQ8Groups = 3;
static_assert(kDkQ8Groups * kQ8GroupBytes <= kDkData, "Q8_0 items fit the stage");
// GGUF Q2_K gate/up: super-blocks of 256 rows of 2688 bytes, four per routed item
constexpr int kDkQ2kSbs = 4;
static_assert(kDkQ2kSbs * kQ2kSbBytes <= kDkData, "Q2_K items fit the stage");
// GGUF Q4_K gate/up: super-blocks of 4736 bytes, three per routed item
constexpr int kDkQ4kSbs = 3;
static_assert(kDkQ4kSbs * kQ4kSbBytes <= kDkData, "Q4_K items fit the stage");
// draft expert formats (template argument of the launch): INT4, INT4 with zero
// points, GGUF Q8_0, and GGUF Q2_K or Q4_K gate/up with a Q8_0 down projection
enum : int { DK_FMT_W4 = 0, DK_FMT_W4Z = 1, DK_FMT_Q8 = 2, DK_FMT_Q2K = 3, DK_FMT_Q4K = 4 };
__host__ __device__ inline bool dk_kquant(int fmt) { return fmt == DK_FMT_Q2K || fmt == DK_FMT_Q4K; }
constexpr int kDkSdSteps = 16;    // k-steps of I_s per SD item
constexpr int kDkMaxStages = 16;  // ring stages (and gate/up slots) at most
constexpr int kDkDBatch = 2;      // down items per queue unit
constexpr int kDkShards = 8;      // independent queue counters (SM b uses shard b % kDkShards)
constexpr uint32_t kDkSleepNs = 1000;  // longest sleep of a waiting warp inside one try_wait
// Warp roles.  An SM's four sub-partitions (each with its own scheduler,
// instruction cache and tensor pipe) take warps by index mod 4.  The producer
// (warp 3) and the poller (warp 7) have sub-partition 3 to themselves (warp
// 11, when the block has one, does nothing): a consumer warp there took the
// issue slots from the producer, whose per-unit work then ran several times
// slower.  The consumer warps fill sub-partitions 0-2.  The warps of a
// sub-partition share its 16K registers (kDkMaxRegs per thread).
constexpr int kDkCons = 9;
constexpr int kDkWarps = 11;
constexpr int kDkProducerWarp = 3, kDkPollerWarp = 7;
constexpr int kDkIdleWarp = kDkWarps > 12 ? 11 : -1;  // keeps sub-partition 3 to the producer and the poller
constexpr int kDkIdleWarp2 = -1;
constexpr int kDkThreads = kDkWarps * 32;
constexpr int kDkMaxRegs = (65536 / (((kDkWarps + 3) / 4) * 4 * 32) / 8 * 8) < 168
                               ? 65536 / (((kDkWarps + 3) / 4) * 4 * 32) / 8 * 8
                               : 168;
__host__ __device__ constexpr bool dk_not_consumer(int w) {
    return w == kDkProducerWarp || w == kDkPollerWarp || w == kDkIdleWarp || w == kDkIdleWarp2;
}
// consumer index 0..kDkCons-1 of a consumer warp: the consumer warps below it
__host__ __device__ constexpr int dk_consumer_index(int warp) {
    int c = 0;
    for (int w = 0; w < warp; ++w) c += dk_not_consumer(w) ? 0 : 1;
    return c;
}
static_assert(kDkWarps > kDkPollerWarp && kDkWarps > kDkProducerWarp &&
                  kDkCons == kDkWarps - 2 - (kDkIdleWarp >= 0 ? 1 : 0) - (kDkIdleWarp2 >= 0 ? 1 : 0),
              "consumer warps");
static_assert(kDkMaxRegs >= 64, "registers per thread of the draft launch");

struct __align__(16) DHeader {
    int kind;
    int a;       // active slot (routed items)
    int e;       // expert (routed items)
    int blk;     // SG: shared block; RG: slice; SD/RD: output pair
    int r;       // range index
    int k0;      // SG: first k-step of H; RG: first group of H; SD: first k-step of I_s; RD: first group of I
    int n;       // SG/SD: k-steps; RG/RD: groups
    int seq;     // ring sequence number of this stage fill
    int slot;    // gate/up: shared-memory slot of the column block
    int nitems;  // gate/up: items of the column block
    int bseq;    // gate/up: column-block sequence number on this SM
    int hpar;    // down items: phase parity of the stage's h-slice barrier for this fill
};

// A down item's h slice that the poller copies once the slice is complete.
struct DPend {
    const void *src;
    const int *rdy;
    int target;
    uint32_t bytes;
    unsigned long long t_reg;  // profiling build: when the producer registered it
};

struct DkGeom {
    int sg_cols, sg_nks, sg_nr;  // shared gate/up: blocks of 16 columns, k-steps per item, items per block
    int sd_nr;                   // shared down ranges of kDkSdSteps k-steps
    int rg_blocks, rg_gpi, rg_nr;
    int rd_gpi, rd_nr;  // routed down: groups per item, ranges
};

// fmt: DK_FMT_*; the GGUF formats use S = 16, K-quant gate/up items count
// super-blocks of 256 rows instead of groups of 128.
__host__ __device__ inline DkGeom dk_geom(int H, int I, int S, int I_s, int fmt = DK_FMT_W4) {
    const bool q8dn = fmt == DK_FMT_Q8 || dk_kquant(fmt);
    DkGeom g;
    g.sg_cols = I_s / 16;
    g.sg_nks = ((H / 16) % 16 == 0) ? 16 : 8;
    g.sg_nr = (H / 16) / g.sg_nks;
    g.sd_nr = (I_s / 16 + kDkSdSteps - 1) / kDkSdSteps;
    g.rg_blocks = I / S;
    g.rg_gpi = fmt == DK_FMT_Q8    ? kDkQ8Groups
               : fmt == DK_FMT_Q2K ? kDkQ2kSbs
               : fmt == DK_FMT_Q4K ? kDkQ4kSbs
                                   : (S == 32 ? 4 : 8);
    g.rg_nr = (H / (dk_kquant(fmt) ? 256 : 128) + g.rg_gpi - 1) / g.rg_gpi;
    g.rd_gpi = q8dn ? kDkQ8Groups : kDkRdGroups;
    g.rd_nr = (I / 128 + g.rd_gpi - 1) / g.rd_gpi;
    return g;
}

// Scratch in the workspace (after the token tables), 256-byte aligned parts:
// the intermediates h (B-fragment order) and the per-range ready counts.
struct DkScratch {
    size_t qctr, hf_s, hf_r, rdy_s, rdy_r, end;
};
__host__ __device__ inline size_t al256(size_t v) { return (v + 255) / 256 * 256; }
__host__ __device__ inline DkScratch dk_scratch(size_t base, int T, int H, int I, int I_s, int nact_max) {
    const DkGeom g = dk_geom(H, I, 16, I_s, DK_FMT_Q8);  // the format with the most down ranges
    static_assert(kDkQ8Groups <= kDkRdGroups, "ready counts sized for the smallest down items");
    DkScratch s;
    size_t o = al256(base);
    s.qctr = o;  // one 256-byte line per queue shard
    o += (size_t)kDkShards * 256;
    s.hf_s = o;
    o = al256(o + (size_t)(I_s / 16) * T * 32);
    s.hf_r = o;
    o = al256(o + (size_t)nact_max * (I / 16) * T * 32);
    s.rdy_s = o;
    o = al256(o + (size_t)g.sd_nr * 4);
    s.rdy_r = o;
    o = al256(o + (size_t)nact_max * g.rd_nr * 4);
    s.end = o;
    return s;
}

// Shared memory.  One gate/up slot per ring stage: a column block holds at
// least one stage until it completes, so slots never run out before stages.
struct DkLayout {
    int bars, hdrs, misc, gamma, act, sfree, scnt, pstate, pend, sacc, rids, rpw, rrank, rsv, stn, ste, sx, sx16, xs,
        ring, stage, hs_off, total, xs_stride, slot_floats;
};
// kq: room for the x sums of GGUF K-quant gate/up items (hi, lo fp16; over 16
// rows for Q2_K, 32 rows for Q4_K).
__host__ __device__ inline DkLayout dk_layout(int T, int H, int nst, int k, int nact_max, int E, bool kq = false) {
    DkLayout L;
    int o = 0;
    L.bars = o;  // full[nst] (weights), empty[nst], hfull[nst] (h slices), all-consumer barrier, routing barrier
    o += (3 * nst + 2) * 8;
    o = (o + 15) & ~15;
    L.hdrs = o;
    o += nst * (int)sizeof(DHeader);
    L.misc = o;
    o += 64;
    L.gamma = o;
    o += kMaxT * 4;
    L.act = o;
    o += kMaxE * 4;
    L.sfree = o;
    o += kDkMaxStages * 4;
    L.scnt = o;
    o += kDkMaxStages * 4;
    L.pstate = o;
    o += kDkMaxStages * 4;
    o = (o + 15) & ~15;
    L.pend = o;
    o += kDkMaxStages * (int)sizeof(DPend);
    L.sacc = o;
    L.slot_floats = 2 * 32 * T;  // [gate|up][32 columns][T]
    o += nst * L.slot_floats * 4;
    // routing of the launch's tokens: selections, counting sort, token tables
    L.rids = o;
    o += T * k * 4;
    L.rpw = o;
    o += T * k * 4;
    L.rrank = o;
    o += T * k * 4;
    o = (o + 15) & ~15;
    L.rsv = o;  // per selecting warp (one per token): the token's logits
    o += T * E * 4;
    L.stn = o;
    o += nact_max * 4;
    o = (o + 15) & ~15;
    L.ste = o;
    o += nact_max * T * (int)sizeof(TokEntry);
    L.sx = o;  // [T][H/128] group sums of x (fp32)
    o += T * (H / 128) * 4;
    o = (o + 15) & ~15;
    L.sx16 = o;  // Q2_K: [T][H/16] sums of x over 16 rows, fp16 hi, then lo (Q4_K: [T][H/32] each)
    o += kq ? T * (H / 16) * 4 : 0;
    o = (o + 15) & ~15;
    L.xs = o;
    L.xs_stride = H + 8;
    o += T * (H + 8) * 2;
    o = (o + 127) & ~127;
    L.ring = o;
    L.hs_off = kDkData;
    const int hs_bytes = ((kDkRdGroups * 8 > kDkSdSteps ? kDkRdGroups * 8 : kDkSdSteps) * T * 32 + 127) & ~127;
    L.stage = kDkData + hs_bytes;
    o += nst * L.stage;
    L.total = o;
    return L;
}

struct DkParams {
    const uint8_t *w4;      // packed INT4 (or Q8_0) experts
    int fmt;                // DK_FMT_* of the routed experts
    const __half *zeros_gu, *zeros_dn;  // nullable: per-group zero points (else 8), repacked
    size_t w4_colblk;       // byte offset of the column-block-major down weights
    int S;                  // INT4 slice width
    const uint8_t *sh;      // shared pack (nullable)
    const __half *w_sgate;  // nullable
    int I_s;
    int E, I, k, T, H;
    const int32_t *active, *n_active;
    const TokTable *tables;
    const __half *x;
    int mode;  // 0: rows of y_sorted, scale 1; 2: weighted into the fp32 accumulator, last block writes out
    // routing inside the launch (logits != nullptr) and its outputs (block 0)
    const float *logits;
    int renorm;
    int32_t *topk_ids;
    float *topk_w;
    uint32_t *elb;
    int layer;
    int32_t *counts, *offsets, *sorted_slots, *active_out, *n_active_out;
    float *yout;
    __half *out;
    WsHeader *hdr;
    uint32_t *qctr;  // queue shard s counter at qctr[64 * s]
    uint2 *hf_s, *hf_r;
    int *rdy_s, *rdy_r;
    int nact_max, nstages;
    uint64_t wait_budget_ns;
    int tl_slot;  // profiling build: slot of this launch's phase marks
};

// Like mbar_try_wait, but the thread may sleep up to `ns` in the wait (it
// wakes as soon as the phase completes), so waiting warps leave the issue
// slots to the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                        int32_t *status, uint64_t budget_ns,
                                                        int32_t site = SITE_HSLICE) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait_sleep(bar, parity, kDkSleepNs)) return true;
        if (global_timer_ns() - t0 > budget_ns) {
            record_timeout(status, site);
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ int ld_relaxed_gpu(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// misc words: [0] abort flag, [1] last-block flag, [2] consumer stage ticket,
// [3] producer has registered its last h copy, [4] routing is in shared
// memory, [5] number of active experts.

// ------------------------------------------------------------- producer --
// One ring fill as a producer lane describes it: the stage header, the
// weights (and zero points) to copy, and for a down item the h slice the
// poller copies once it is complete.
struct DFill {
    DHeader h;
    const uint8_t *src;
    const void *zsrc, *hsrc;
    const int *rdy;
    uint32_t bytes, zbytes, zoff, hs_bytes;
    int target;
};

// Queue tickets: [shared gate/up blocks][routed gate/up blocks][down items in
// pairs].  Every gate/up block is dequeued before any down item, and a block's
// items enter this SM's ring before anything it dequeues later, so h always
// completes: the down items that wait for it never hold up a gate/up item.
//
// The whole producer warp runs this: lane j describes fill j of the current
// queue unit, and up to min(stages, 16) lanes issue their fills at once, so
// the serial work per fill is the copy issue itself (a lone thread spent ~0.4
// us of address arithmetic per fill).  Lane 0 takes the queue tickets.
__device__ void dk_producer(const DkParams &p, uint8_t *smem, const DkLayout &L, int lane) {
    constexpr unsigned kAll = 0xffffffffu;
    const int nst = p.nstages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + nst;
    uint64_t *hfull = empty + nst;
    DHeader *hdrs = reinterpret_cast<DHeader *>(smem + L.hdrs);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L.misc);
    const int *act = reinterpret_cast<const int *>(smem + L.act);
    volatile int *sfree = reinterpret_cast<volatile int *>(smem + L.sfree);
    volatile int *pstate = reinterpret_cast<volatile int *>(smem + L.pstate);
    DPend *pend = reinterpret_cast<DPend *>(smem + L.pend);
    uint8_t *ring = smem + L.ring;
    const uint64_t pol = policy_evict_first();
    const int H = p.H, I = p.I, T = p.T;
    const DkGeom g = dk_geom(H, I, p.S, p.I_s, p.fmt);
    const bool q8dn = p.fmt == DK_FMT_Q8 || dk_kquant(p.fmt);
    const int NQ = H / 32;
    const int nSGb = p.sh ? g.sg_cols : 0;
    const int nSD = p.sh ? NQ * g.sd_nr : 0;
    const int ngroups = H / (dk_kquant(p.fmt) ? 256 : 128);  // gate/up groups (K-quant: super-blocks) of H
    const size_t rg_gb = p.fmt == DK_FMT_Q8    ? (size_t)kQ8GroupBytes
                         : p.fmt == DK_FMT_Q2K ? (size_t)kQ2kSbBytes
                         : p.fmt == DK_FMT_Q4K ? (size_t)kQ4kSbBytes
                                               : w4_group_bytes(p.S);
    const size_t rg_ub = p.fmt == DK_FMT_Q8    ? q8_unit_bytes(H)
                         : p.fmt == DK_FMT_Q2K ? q2k_unit_bytes(H)
                         : p.fmt == DK_FMT_Q4K ? q4k_unit_bytes(H)
                                               : w4_unit_bytes(H, p.S);
    const uint32_t rd_gb = q8dn ? (uint32_t)kQ8GroupBytes : (uint32_t)kW4ColGroupBytes;
    const int wmax = nst < 16 ? nst : 16;  // fills issued per round: distinct stages
    bool ok = true;                        // warp-uniform
    int na = -1;
    uint32_t it = 0;         // fills issued so far
    uint32_t hpar_bits = 0;  // bit st: phase parity of hfull[st] for the stage's next down fill
    int bseq = 0;            // gate/up column blocks taken so far
    // A bounded wait gave up: record it once and raise the block's abort flag.
    auto timed_out = [&](int32_t site) {
        if (lane == 0) {
            record_timeout(&p.hdr->status, site);
            misc[0] = 1;
        }
        ok = false;
    };
    auto expired = [&](uint64_t t0) { return __any_sync(kAll, global_timer_ns() - t0 > p.wait_budget_ns); };
    // Shared words other warps write are read by lane 0 and broadcast: every
    // lane then takes the same branch, so the lanes of this warp always meet
    // at the same collective (lanes that read such a word each for itself can
    // see different values and drift apart).
    auto rd0 = [&](const volatile int *w) {
        int v = 0;
        if (lane == 0) v = *w;
        return __shfl_sync(kAll, v, 0);
    };
    // Active experts: the consumer warps route the launch's tokens into shared
    // memory at start; routed work waits for that (shared gate/up does not).
    // The routing barrier completes once per launch; every lane waits on it
    // (a suspended wait that resumes as soon as the routing warp arrives).
    uint64_t *rbar = hfull + nst + 1;
    auto n_act = [&]() -> int {
        if (na < 0) {
            const uint64_t t0 = global_timer_ns();
            while (true) {
                const bool seen = mbar_try_wait_sleep(rbar, 0, kDkSleepNs);
                if (__all_sync(kAll, seen)) break;
                if (rd0(misc)) {
                    ok = false;
                    return na = 0;
                }
                if (expired(t0)) {
                    timed_out(SITE_ROUTING);
                    return na = 0;
                }
            }
            na = rd0(misc + 5);
        }
        return na;
    };
    // Slot of the next gate/up column block (its partial sums meet there).
    auto take_slot = [&](DHeader &h, int nitems) -> bool {
        const int slot = bseq % nst;
        if (rd0(sfree + slot) != bseq) {  // the slot's previous block is still being completed
            const uint64_t t0 = global_timer_ns();
            while (rd0(sfree + slot) != bseq) {
                if (rd0(misc)) {
                    ok = false;
                    return false;
                }
                if (expired(t0)) {
                    timed_out(SITE_SLOT);
                    return false;
                }
                __nanosleep(64);
            }
        }
        h.slot = slot;
        h.nitems = nitems;
        h.bseq = bseq++;
        return true;
    };
    // Issues fills 0..n-1 of the unit (lane j holds fill j), in rounds of at
    // most wmax lanes (distinct stages); within a round each lane issues its
    // fill as soon as its own stage is free.
    auto issue_fills = [&](const DFill &f, int n) -> bool {
        __syncwarp();  // lanes that finished describing their fill early wait here
        for (int base = 0; base < n; base += wmax) {
            const int cnt = min(wmax, n - base);
            const bool mine = lane >= base && lane < base + cnt;
            const uint32_t fi = it + (uint32_t)(lane - base);
            const int st = mine ? (int)(fi % (uint32_t)nst) : 0;
            const uint32_t par = ((fi / (uint32_t)nst) & 1u) ^ 1u;
            const uint32_t tr_w = TR_NOW();
            bool done = !mine;
            uint64_t t0 = 0;
            bool waited = false;
            while (true) {
                const bool go = !done && (waited ? mbar_try_wait_sleep(&empty[st], par, kDkSleepNs)
                                                 : mbar_try_wait(&empty[st], par));
                const bool hs = go && f.hs_bytes;
                if (go) {
                    DHeader h = f.h;
                    h.seq = (int)fi;
                    h.hpar = (int)((hpar_bits >> st) & 1u);
                    hdrs[st] = h;
                    uint8_t *dst = ring + (size_t)st * L.stage;
                    mbar_arrive_expect_tx(&full[st], f.bytes + f.zbytes);
                    if (f.bytes) bulk_g2s(dst, f.src, f.bytes, &full[st], pol);
                    if (f.zbytes) bulk_g2s(dst + f.zoff, f.zsrc, f.zbytes, &full[st], pol);
                    if (hs) {
                        mbar_arrive_expect_tx(&hfull[st], f.hs_bytes);  // completed by the poller's copy
                        pend[st].src = f.hsrc;
                        pend[st].rdy = f.rdy;
                        pend[st].target = f.target;
                        pend[st].bytes = f.hs_bytes;
                        pend[st].t_reg = TL_NOW();
                    }
                    done = true;
                }
                const uint32_t hmask = __reduce_or_sync(kAll, hs ? (1u << st) : 0u);
                if (hmask) {
                    __threadfence_block();  // the pending entries before their flags
                    if (hs) pstate[st] = 1;
                    hpar_bits ^= hmask;
                }
                if (__all_sync(kAll, done)) break;
                if (!waited) {
                    waited = true;
                    t0 = global_timer_ns();
                }
                // giving up: the fills this round did issue land (bounded) before the block may exit
                auto drain_round = [&]() {
                    if (mine && done) {
                        const uint64_t td = global_timer_ns();
                        while (!mbar_try_wait(&full[st], (fi / (uint32_t)nst) & 1u) &&
                               global_timer_ns() - td < 100000000ull) {
                        }
                    }
                };
                if (rd0(misc)) {
                    drain_round();
                    ok = false;
                    return false;
                }
                if (expired(t0)) {
                    timed_out(SITE_STAGE);
                    drain_round();
                    return false;
                }
            }
            const uint32_t tr_r = TR_NOW();
#if TL_ON
            if (mine && TR_ON() && fi < (uint32_t)kTrFills) {
                s_tr.fill[fi][0] = tr_w;
                s_tr.fill[fi][1] = tr_r;
                s_tr.fill[fi][2] = TR_NOW();
                s_tr.fill[fi][3] = ((uint32_t)f.h.kind << 24) | ((f.bytes + f.zbytes) & 0xffffffu);
            }
#else
            (void)tr_w;
            (void)tr_r;
#endif
            it += (uint32_t)cnt;
            if (lane == 0) misc[14] = (int)it;  // fills issued (read when a wait gives up)
        }
        return true;
    };
    // Fills of queue unit u, lane j describing fill j: the fill count, 0 to
    // skip the unit, -1 once the queue is exhausted (or on failure).
    auto expand = [&](int u, DFill &f) -> int {
        if (u < 0) return -1;  // a corrupted queue counter (workspace not zeroed): stop
        f = DFill{};
        if (u < nSGb) {
            DHeader h{};
            h.kind = DK_SG;
            h.blk = u;
            if (!take_slot(h, g.sg_nr)) return -1;
            h.r = lane;
            h.k0 = lane * g.sg_nks;
            h.n = g.sg_nks;
            f.h = h;
            f.src = p.sh + (size_t)h.blk * f16_unit_bytes(H) + (size_t)h.k0 * 1024;
            f.bytes = (uint32_t)h.n * 1024;
            return g.sg_nr;
        }
        int v = u - nSGb;
        const int nA = n_act();
        if (!ok) return -1;
        const int nRGb = nA * g.rg_blocks;
        if (v < nRGb) {
            DHeader h{};
            h.kind = DK_RG;
            h.a = v / g.rg_blocks;
            h.blk = v - h.a * g.rg_blocks;
            h.e = act[h.a];
            if (h.e < 0 || h.e >= p.E) return 0;  // unusable routing entry
            if (!take_slot(h, g.rg_nr)) return -1;
            const size_t unit = (size_t)h.e * g.rg_blocks + h.blk;
            h.r = lane;
            h.k0 = lane * g.rg_gpi;
            h.n = min(g.rg_gpi, ngroups - h.k0);
            f.h = h;
            f.src = p.w4 + unit * rg_ub + (size_t)h.k0 * rg_gb;
            f.bytes = (uint32_t)(h.n * rg_gb);
            if (p.zeros_gu) {  // zero points (2S per group, as the scales) in the stage's h area, unused by these items
                f.zsrc = p.zeros_gu + (unit * (H / 128) + h.k0) * 2 * p.S;
                f.zbytes = (uint32_t)h.n * 4u * (uint32_t)p.S;
                f.zoff = (uint32_t)L.hs_off;
            }
            return g.rg_nr;
        }
        v -= nRGb;
        const int nRD = nA * NQ * g.rd_nr;
        const int d0 = v * kDkDBatch;
        if (d0 >= nSD + nRD) return -1;
        const int n = min(kDkDBatch, nSD + nRD - d0);
        int d = d0 + lane;
        if (lane >= n) return n;
        DHeader h{};
        if (d < nSD) {
            h.kind = DK_SD;
            h.r = d / NQ;
            h.blk = d - h.r * NQ;
            h.k0 = h.r * kDkSdSteps;
            h.n = min(kDkSdSteps, p.I_s / 16 - h.k0);
            f.h = h;
            f.src = p.sh + shared_pairdown_offset(H, p.I_s) + ((size_t)h.blk * (p.I_s / 16) + h.k0) * 1024;
            f.bytes = (uint32_t)h.n * 1024;
            f.hsrc = p.hf_s + (size_t)h.k0 * T * 4;
            f.hs_bytes = (uint32_t)(h.n * T * 32);
            f.rdy = p.rdy_s + h.r;
            f.target = h.n;
            return n;
        }
        d -= nSD;
        h.kind = DK_RD;
        h.a = d / (NQ * g.rd_nr);
        const int rem = d - h.a * (NQ * g.rd_nr);
        h.r = rem / NQ;
        h.blk = rem - h.r * NQ;
        h.e = act[h.a];
        if (h.e < 0 || h.e >= p.E) {  // unusable routing entry: an empty fill the consumer skips
            h.kind = DK_NOP;
            f.h = h;
            return n;
        }
        h.k0 = h.r * g.rd_gpi;
        h.n = min(g.rd_gpi, I / 128 - h.k0);
        f.h = h;
        f.src = p.w4 + p.w4_colblk + (((size_t)h.e * NQ + h.blk) * (I / 128) + h.k0) * rd_gb;
        f.bytes = (uint32_t)h.n * rd_gb;
        f.hsrc = p.hf_r + ((size_t)h.a * (I / 16) + (size_t)h.k0 * 8) * T * 4;
        f.hs_bytes = (uint32_t)(h.n * 8 * T * 32);
        f.rdy = p.rdy_r + h.a * g.rd_nr + h.r;
        f.target = h.n * 8;
        if (p.zeros_dn) {
            f.zsrc = p.zeros_dn + (((size_t)h.e * NQ + h.blk) * (I / 128) + h.k0) * 32;
            f.zbytes = (uint32_t)h.n * 64u;
            f.zoff = (uint32_t)kDkRdZeroOff;
        }
        return n;
    };
    int tr_nunit = 0;
    DFill f;
    auto run_unit = [&](int u) -> bool {
#if TL_ON
        if (lane == 0 && TR_ON() && tr_nunit < kTrUnits) {
            s_tr.unit[tr_nunit][0] = TR_NOW();
            s_tr.unit[tr_nunit][1] = (uint32_t)u;
        }
        ++tr_nunit;
#else
        (void)tr_nunit;
#endif
        const int n = expand(u, f);
#if TL_ON
        if (lane == 0 && TR_ON() && tr_nunit <= kTrUnits) s_tr.unit[tr_nunit - 1][2] = TR_NOW();
#endif
        if (n < 0) return false;
        const bool r = n == 0 || issue_fills(f, n);
#if TL_ON
        if (lane == 0 && TR_ON() && tr_nunit <= kTrUnits) s_tr.unit[tr_nunit - 1][3] = TR_NOW();
#endif
        return r;
    };
    // The queue is split into kDkShards interleaved shards (unit u belongs to
    // shard u % kDkShards) so that each counter serves a few SMs only.  Each
    // block's first ticket in its shard is static; two tickets are in flight,
    // so the next dequeue is issued a whole ticket ahead.
    const int shard = (int)(blockIdx.x % kDkShards);
    const uint32_t nsm = (gridDim.x - shard + kDkShards - 1) / kDkShards;  // blocks on this shard
    uint32_t *ctr = p.qctr + 64 * shard;
    // The static unit's fills need no global memory but its weights (the
    // routing and the ready counts are the consumers' and the poller's, who
    // wait for the preceding launch themselves), so they are issued before
    // this warp waits for it; the counters come after.
    // One call site of the unit logic (it is large): the first pass runs the
    // static unit, then waits for the preceding launch; later passes take a
    // ticket that was fetched one unit ahead.
    uint32_t tk = blockIdx.x / kDkShards;  // lane 0: the unit's ticket
    uint32_t tnext = 0;                    // lane 0: the next ticket, in flight
    bool first = true, took = false;
    while (true) {
        const bool more = run_unit((int)__shfl_sync(kAll, tk, 0) * kDkShards + shard);
        if (first) {
            first = false;
            if (lane == 0) TLB_FIRST(p.tl_slot, TL_PROD_STATIC);
            griddep_wait();
            if (lane == 0) TLB_FIRST(p.tl_slot, TL_PROD_GRIDDEP);
            if (!more) break;
            if (lane == 0) tnext = nsm + atomicAdd(ctr, 1u);
            took = true;
        } else if (!more) {
            break;
        }
        if (lane == 0) {
            tk = tnext;  // fetched a whole unit ago
            tnext = nsm + atomicAdd(ctr, 1u);
        }
        __syncwarp();
    }
    // The ticket taken ahead is still in flight: wait for its value (a
    // returned value means the add is done at L2) and fence, so that no add of
    // this block can land after the last block has reset the queue counters
    // for the next call (the end markers only release at block scope).
    if (took && lane == 0) {
        misc[15] = (int)tnext;
        __threadfence();
    }
    if (ok) {
        if (lane == 0) TLB_LAST(p.tl_slot, TL_PROD_LAST);
        __threadfence_block();
        if (lane == 0) misc[3] = 1;  // no more h copies to register
        f = DFill{};                 // one end marker per consumer warp
        f.h.kind = DK_DONE;
        issue_fills(f, kDkCons);
    }
    if (!ok && lane == 0) {
        // bounded wait for the copies in flight before the block may exit
        const uint32_t first = it > (uint32_t)nst ? it - nst : 0;
        for (uint32_t j = first; j < it; ++j) {
            const int st = (int)(j % nst);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[st], (j / nst) & 1) && global_timer_ns() - t0 < 100000000ull) {
            }
        }
    }
}

// --------------------------------------------------------------- poller --
// Copies each pending down item's h slice into its stage once the slice's
// ready count reaches the item's target (a relaxed poll of all pending counts
// at once, then an acquire fence and a proxy fence before the bulk copies).
__device__ void dk_poller(const DkParams &p, uint8_t *smem, const DkLayout &L) {
    const int nst = p.nstages;
    uint64_t *hfull = reinterpret_cast<uint64_t *>(smem + L.bars) + 2 * nst;
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L.misc);
    volatile int *pstate = reinterpret_cast<volatile int *>(smem + L.pstate);
    const DPend *pend = reinterpret_cast<const DPend *>(smem + L.pend);
    const DHeader *hdrs = reinterpret_cast<const DHeader *>(smem + L.hdrs);
    uint8_t *ring = smem + L.ring;
    griddep_wait();  // the ready counts of the preceding launch's workspace use
    uint64_t t_last = global_timer_ns();
    uint32_t issued = 0, ipar = 0;  // copies in flight (bit j) and their hfull phase parity
    // On an abort the block exits early: wait (bounded) for this warp's copies first.
    auto drain = [&]() {
        for (int j = 0; j < nst; ++j) {
            if (!((issued >> j) & 1u)) continue;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&hfull[j], (ipar >> j) & 1u) && global_timer_ns() - t0 < 100000000ull) {
            }
        }
    };
    while (true) {
        if (misc[0]) {
            drain();
            return;
        }
        // forget the copies that have landed
        for (int j = 0; j < nst; ++j)
            if (((issued >> j) & 1u) && mbar_try_wait(&hfull[j], (ipar >> j) & 1u)) issued &= ~(1u << j);
        const int fin = misc[3];
        __threadfence_block();
        uint32_t m = 0;
        for (int j = 0; j < nst; ++j) m |= (pstate[j] == 1 ? 1u : 0u) << j;
        if (!m) {
            if (fin) return;
            __nanosleep(100);
            t_last = global_timer_ns();
            continue;
        }
        __threadfence_block();
        // all pending counts are loaded at once, then the complete slices copied
        int v[kDkMaxStages];
#pragma unroll
        for (int j = 0; j < kDkMaxStages; ++j) v[j] = ((m >> j) & 1u) ? ld_relaxed_gpu(pend[j].rdy) : 0;
        uint32_t go = 0;
#pragma unroll
        for (int j = 0; j < kDkMaxStages; ++j) go |= (((m >> j) & 1u) && v[j] >= pend[j].target ? 1u : 0u) << j;
        const bool any = go != 0;
        if (any) {
            fence_acq_rel_gpu();         // the h stores counted by the ready count
            fence_proxy_async_global();  // ... are read through the bulk-copy proxy
        }
        while (go) {
            const int j = __ffs(go) - 1;
            go &= go - 1;
            bulk_g2s_plain(ring + (size_t)j * L.stage + L.hs_off, pend[j].src, pend[j].bytes, &hfull[j]);
            TL_ADD(p.tl_slot, TL_W_POLL, TL_NOW() - pend[j].t_reg);
            issued |= 1u << j;
            ipar = (ipar & ~(1u << j)) | ((uint32_t)hdrs[j].hpar << j);
            pstate[j] = 0;
        }
        if (any) {
            t_last = global_timer_ns();
        } else if (global_timer_ns() - t_last > p.wait_budget_ns) {
            record_timeout(&p.hdr->status, SITE_POLLER);
            misc[0] = 1;
            drain();
            return;
        }
    }
}

// ------------------------------------------------------------ consumers --
// Completes a column block whose partial sums are all in shared-memory slot
// `sa` ([gate|up][32 columns][T]): h = silu(g) * u for token column t and the
// block's k-steps kk (rows 16 kk + {2q, 2q+1, 2q+8, 2q+9}), packed as B
// fragments (two half2) into hf[kk]; the slot is cleared on the way.
__device__ __forceinline__ void finalize_block(float *sa, int T, int nk, int lane, uint2 *hf, size_t hf_kstride) {
    const int t = lane >> 2, q4 = lane & 3;
    if (t >= T) return;
    const int off[4] = {2 * q4, 2 * q4 + 1, 2 * q4 + 8, 2 * q4 + 9};
    for (int kk = 0; kk < nk; ++kk) {
        float hv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            volatile float *gp = sa + (size_t)(16 * kk + off[j]) * T + t;
            volatile float *up = gp + 32 * T;
            const float gv = *gp, uv = *up;
            *gp = 0.f;
            *up = 0.f;
            hv[j] = gv / (1.0f + __expf(-gv)) * uv;
        }
        uint2 r;
        r.x = h2_as_u32(__floats2half2_rn(hv[0], hv[1]));
        r.y = h2_as_u32(__floats2half2_rn(hv[2], hv[3]));
        hf[(size_t)kk * hf_kstride + (size_t)t * 4 + q4] = r;
    }
}

// Counting sort of the launch's T*k selections by expert, by one warp, into
// shared memory (no shuffles: T*k is small, every lane scans the slot list):
// the active experts in ascending order (act), each active expert's token
// table (ste[a*T + rank]: token s/k, output row s/k, gate weight, in slot
// order; stn[a] entries).  With out (block 0) the gather arrays of the routing
// outputs are written as well.  Returns the number of active experts.
__device__ __noinline__ int route_tables_warp(const DkParams &p, const DkLayout L, uint8_t *smem, int lane,
                                              bool out) {
    const int E = p.E, k = p.k, T = p.T, n = T * k;
    const int32_t *ids = reinterpret_cast<const int32_t *>(smem + L.rids);
    const float *pw = reinterpret_cast<const float *>(smem + L.rpw);
    int *rank = reinterpret_cast<int *>(smem + L.rrank);
    int *act = reinterpret_cast<int *>(smem + L.act);
    int *stn = reinterpret_cast<int *>(smem + L.stn);
    TokEntry *ste = reinterpret_cast<TokEntry *>(smem + L.ste);
    int nfirst = 0;
    for (int s = lane; s < n; s += 32) {  // rank of slot s among the earlier slots of its expert
        const int e = ids[s];
        int r = 0;
        for (int s2 = 0; s2 < s; ++s2) r += (ids[s2] == e);
        rank[s] = r;
        nfirst += (r == 0);
    }
    const int na = __reduce_add_sync(0xffffffffu, nfirst);
    __syncwarp();
    for (int s = lane; s < n; s += 32) {
        const int e = ids[s], r = rank[s];
        int a = 0, c = 0, below = 0;  // active experts below e, slots of e, slots of experts below e
        for (int s2 = 0; s2 < n; ++s2) {
            const int e2 = ids[s2];
            a += (e2 < e && rank[s2] == 0);
            c += (e2 == e);
            below += (e2 < e);
        }
        TokEntry te;
        te.tok = s / k;
        te.row = s / k;
        te.scale = pw[s];
        te.pad = 0;
        if (r < T) ste[a * T + r] = te;  // an expert holds at most one slot per token
        if (r == 0) {
            act[a] = e;
            stn[a] = c;
        }
        if (out) p.sorted_slots[below + r] = s;
    }
    if (out) {
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            int c = 0, below = 0;
            for (int s2 = 0; s2 < n; ++s2) {
                c += (ids[s2] == e);
                below += (ids[s2] < e);
            }
            p.counts[e] = c;
            p.offsets[e] = below;
            p.active_out[e] = e < na ? act[e] : -1;
        }
        if (lane == 0) {
            p.offsets[E] = n;
            *p.n_active_out = na;
        }
    }
    return na;
}

// One token, at most 32 selections (every block the same way): its k
// experts straight from the logits in global memory, then the active-expert
// table (an expert's place = the selected experts below it; each holds one
// slot, the token's).  Returns k.  The routing outputs are written apart, by
// route_one_outputs, once the tables are published.
__device__ __noinline__ int route_one_token(const DkParams &p, const DkLayout L, uint8_t *smem, int lane) {
    const int E = p.E, k = p.k;
    int32_t *ids = reinterpret_cast<int32_t *>(smem + L.rids);
    float *pw = reinterpret_cast<float *>(smem + L.rpw);
    select_token_global(p.logits, E, k, p.renorm, lane, ids, pw);
#if TL_ON
    if (lane == 0 && TR_ON()) s_tr.route[1] = TR_NOW();
#endif
    int *act = reinterpret_cast<int *>(smem + L.act);
    int *stn = reinterpret_cast<int *>(smem + L.stn);
    TokEntry *ste = reinterpret_cast<TokEntry *>(smem + L.ste);
    const int e = lane < k ? ids[lane] : 0x7fffffff;
    int a = 0;
    for (int s2 = 0; s2 < k; ++s2) a += __shfl_sync(0xffffffffu, e, s2) < e;
    if (lane < k) {
        TokEntry te;
        te.tok = 0;
        te.row = 0;
        te.scale = pw[lane];
        te.pad = 0;
        ste[a] = te;
        act[a] = e;
        stn[a] = 1;
    }
    return k;
}

// Block 0's routing outputs for one token (k <= 32): the selections and
// their weights, the lookahead counters, and the gather arrays (per-expert
// counts and offsets, slots in expert order, the active list).
__device__ __noinline__ void route_one_outputs(const DkParams &p, const DkLayout L, const uint8_t *smem, int lane) {
    const int E = p.E, k = p.k;
    const int32_t *ids = reinterpret_cast<const int32_t *>(smem + L.rids);
    const float *pw = reinterpret_cast<const float *>(smem + L.rpw);
    const int *act = reinterpret_cast<const int *>(smem + L.act);
    const int e = lane < k ? ids[lane] : 0x7fffffff;
    if (lane < k) {
        int a = 0;
        for (int s2 = 0; s2 < k; ++s2) a += ids[s2] < e;
        p.topk_ids[lane] = e;
        p.topk_w[lane] = pw[lane];
        p.sorted_slots[a] = lane;
        if (p.elb) atomicAdd(p.elb + (size_t)p.layer * E + e, 1u);
    }
    for (int e2 = lane; e2 < E; e2 += 32) {
        int c = 0, below = 0;
        for (int s2 = 0; s2 < k; ++s2) {
            const int es = ids[s2];
            c += es == e2;
            below += es < e2;
        }
        p.counts[e2] = c;
        p.offsets[e2] = below;
        p.active_out[e2] = e2 < k ? act[e2] : -1;
    }
    if (lane == 0) {
        p.offsets[E] = k;
        *p.n_active_out = k;
    }
}

// The unit call's routing: active experts and their token tables from global
// memory (written by the preceding launches), into shared memory.
__device__ __noinline__ int load_tables_warp(const DkParams &p, const DkLayout L, uint8_t *smem, int lane) {
    const int T = p.T;
    int *act = reinterpret_cast<int *>(smem + L.act);
    int *stn = reinterpret_cast<int *>(smem + L.stn);
    TokEntry *ste = reinterpret_cast<TokEntry *>(smem + L.ste);
    griddep_wait();
    const int v = __ldcg(p.n_active);
    const int na = v < 0 ? 0 : (v > p.nact_max ? p.nact_max : v);
    for (int a = lane; a < na; a += 32) act[a] = __ldcg(p.active + a);
    __syncwarp();
    for (int i = lane; i < na * T; i += 32) {
        const int a = i / T, j = i - a * T;
        const int e = act[a];
        if (e < 0 || e >= p.E) continue;  // skipped by the producer
        if (j == 0) stn[a] = min(max(__ldcg(&p.tables[e].n), 0), T);
        TokEntry te;
        te.tok = __ldcg(&p.tables[e].e[j].tok);
        te.row = __ldcg(&p.tables[e].e[j].row);
        te.scale = __ldcg(&p.tables[e].e[j].scale);
        te.pad = 0;
        ste[i] = te;
    }
    return na;
}

// INT4 draft kernel; MS = S/16 of the packed INT4 units.
template <int MS, int FMT>
__global__ void __maxnreg__(kDkMaxRegs) draft_kernel(const DkParams p) {
    constexpr bool ZP = FMT == DK_FMT_W4Z;  // INT4 with per-group zero points
    constexpr bool Q8 = FMT == DK_FMT_Q8;   // GGUF Q8_0 (S = 16)
    constexpr bool Q2K = FMT == DK_FMT_Q2K; // GGUF Q2_K gate/up, Q8_0 down (S = 16)
    constexpr bool Q4K = FMT == DK_FMT_Q4K; // GGUF Q4_K gate/up, Q8_0 down (S = 16)
    constexpr bool Q8DN = Q8 || Q2K || Q4K; // Q8_0 down items
    static_assert(!Q8DN || MS == 1, "GGUF experts use 16-column slices");
    extern __shared__ __align__(128) uint8_t smem[];
    // A launch that follows on the stream may be scheduled as SMs free up; it
    // reads nothing of this one before its own griddepcontrol.wait.
    griddep_launch_dependents();
    TL_INIT();
    const int nst = p.nstages;
    const DkLayout L = dk_layout(p.T, p.H, nst, p.k, p.nact_max, p.E, Q2K || Q4K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q4 = lane & 3;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + nst;
    uint64_t *hfull = empty + nst;
    uint64_t *allbar = hfull + nst;
    uint64_t *rbar = allbar + 1;  // routing published (one arrival, by the routing warp)
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    int *scnt = reinterpret_cast<int *>(smem + L.scnt);
    volatile int *sfree = reinterpret_cast<volatile int *>(smem + L.sfree);
    float *sacc = reinterpret_cast<float *>(smem + L.sacc);
    for (int i = threadIdx.x; i < nst * L.slot_floats; i += kDkThreads) sacc[i] = 0.f;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&hfull[s], 1);
        }
        mbar_init(allbar, kDkCons);
        mbar_init(rbar, 1);
        for (int i = 0; i < 16; ++i) misc[i] = 0;
        int *pstate = reinterpret_cast<int *>(smem + L.pstate);
        for (int s = 0; s < kDkMaxStages; ++s) {
            sfree[s] = s;  // slot s first takes block s
            scnt[s] = 0;
            pstate[s] = 0;
        }
        DHeader *hw = reinterpret_cast<DHeader *>(smem + L.hdrs);
        for (int st = 0; st < nst; ++st) hw[st].seq = -1;  // no fill yet (shared memory is not cleared)
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) TLB_FIRST(p.tl_slot, TL_ENTRY);
    if (warp == kDkProducerWarp) {
        dk_producer(p, smem, L, lane);
        return;
    }
    if (warp == kDkPollerWarp) {
        if (lane == 0) dk_poller(p, smem, L);
        return;
    }
    if (warp == kDkIdleWarp || warp == kDkIdleWarp2) return;
    const int cw = dk_consumer_index(warp);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc);
    uint32_t allphase = 0;
    // Consumer barrier; a waiting warp sleeps in the wait (it leaves the
    // issue slots and shared memory to the warps the others wait for).
    auto all_sync = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(allbar);
        mbar_wait_sleep_bounded(allbar, allphase & 1, abort_flag, &p.hdr->status, p.wait_budget_ns, SITE_ALL_SYNC);
        allphase ^= 1;
        __syncwarp();
    };
    const DHeader *hdrs = reinterpret_cast<const DHeader *>(smem + L.hdrs);
    const uint8_t *ring = smem + L.ring;
    float *gamma = reinterpret_cast<float *>(smem + L.gamma);
    __half *xs = reinterpret_cast<__half *>(smem + L.xs);
    const int H = p.H, I = p.I, T = p.T, xstr = L.xs_stride;
    const int ctid = cw * 32 + lane;
    const DkGeom geo = dk_geom(H, I, p.S, p.I_s, FMT);
    griddep_wait();  // x, the logits and the workspace may come from the preceding launch
    // Routing outputs in shared memory are complete: publish them to the
    // producer (misc[4]) and to the routed items.
    auto publish_routing = [&](int na) {
        __syncwarp();
        if (lane == 0) {
            misc[5] = na;
            __threadfence_block();
            *reinterpret_cast<volatile int *>(misc + 4) = 1;
            mbar_arrive(rbar);  // wakes the producer's routing wait at once
            TLB_FIRST(p.tl_slot, TL_ROUTED);
        }
    };
    // One token with given logits: warp 0 selects its experts at once,
    // straight from the logits in global memory, while the other warps stage
    // x; it arrives on the x barrier first (it stages none) and waits on it
    // after the routing is published.
    const bool route1 = p.logits && T == 1;
    if (route1 && cw == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(allbar);
#if TL_ON
        if (lane == 0 && TR_ON()) s_tr.route[0] = TR_NOW();
#endif
        if (p.k <= 32) {
            publish_routing(route_one_token(p, L, smem, lane));
#if TL_ON
            if (lane == 0 && TR_ON()) s_tr.route[3] = TR_NOW();
#endif
            if (blockIdx.x == 0) route_one_outputs(p, L, smem, lane);  // off the routed items' path
        } else {
            int32_t *rids = reinterpret_cast<int32_t *>(smem + L.rids);
            float *rpw = reinterpret_cast<float *>(smem + L.rpw);
            const int E = p.E, k = p.k;
            select_token_global(p.logits, E, k, p.renorm, lane, rids, rpw);
            if (blockIdx.x == 0)
                for (int r = lane; r < k; r += 32) {
                    const int e = rids[r];
                    p.topk_ids[r] = e;
                    p.topk_w[r] = rpw[r];
                    if (p.elb) atomicAdd(p.elb + (size_t)p.layer * E + e, 1u);
                }
            publish_routing(route_tables_warp(p, L, smem, lane, blockIdx.x == 0));
        }
#if TL_ON
        if (lane == 0 && TR_ON()) s_tr.route[4] = TR_NOW();
#endif
    }

    // x into shared memory, and its sums over each group of 128 (16 chunks of
    // 8 = one half-warp, as the stride is a multiple of 16 chunks)
    float *sxs = reinterpret_cast<float *>(smem + L.sx);
    const int xw = route1 ? cw - 1 : cw, nxw = route1 ? kDkCons - 1 : kDkCons;  // staging warps
    for (int base = xw * 32; xw >= 0 && base < T * (H / 8); base += nxw * 32) {
        const int idx = base + lane;
        float sum = 0.f;
        if (idx < T * (H / 8)) {
            const int t = idx / (H / 8), h8 = idx - t * (H / 8);
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * H) + h8);
            *reinterpret_cast<uint4 *>(xs + (size_t)t * xstr + h8 * 8) = v;
            const __half2 *vh = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(vh[q]);
                sum += f.x + f.y;
            }
        }
        kquant_x_sums<Q2K, Q4K>(sum, lane, idx, T, H, reinterpret_cast<__half *>(smem + L.sx16));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if ((lane & 15) == 0 && idx < T * (H / 8)) sxs[idx / 16] = sum;  // [t][group]: idx/16 = t*(H/128) + group
    }
    if (route1 && cw == 0) {  // its arrival came first
        mbar_wait_sleep_bounded(allbar, allphase & 1, abort_flag, &p.hdr->status, p.wait_budget_ns, SITE_ALL_SYNC);
        allphase ^= 1;
        __syncwarp();
    } else {
        all_sync();  // x is in shared memory
    }
    if (ctid == 0) TLB_FIRST(p.tl_slot, TL_X_STAGED);
    // Routing of several tokens: warps t < T select token t (every block the
    // same way; block 0 also writes the routing outputs); the last of them
    // builds the token tables and raises misc[4].  The other warps go straight
    // to the shared expert's items, which need no routing.
    if (route1) {
    } else if (p.logits) {
        if (cw < T) {
            int32_t *rids = reinterpret_cast<int32_t *>(smem + L.rids);
            float *rpw = reinterpret_cast<float *>(smem + L.rpw);
            const int E = p.E, k = p.k;
            int mine = 0;
            for (int t = cw; t < T; t += kDkCons, ++mine) {
                const float *lg = p.logits + (size_t)t * E;
                select_token_global(lg, E, k, p.renorm, lane, rids + t * k, rpw + t * k);
                if (blockIdx.x == 0 && lane == 0)
                    for (int r = 0; r < k; ++r) {
                        const int e = rids[t * k + r];
                        p.topk_ids[(size_t)t * k + r] = e;
                        p.topk_w[(size_t)t * k + r] = rpw[t * k + r];
                        if (p.elb) atomicAdd(p.elb + (size_t)p.layer * E + e, 1u);
                    }
            }
            int done = 0;
            if (lane == 0) {
                __threadfence_block();
                done = atomicAdd(misc + 6, mine) + mine;
            }
            done = __shfl_sync(0xffffffffu, done, 0);
            if (done == T) {  // every token is selected: build the tables
                __threadfence_block();
                publish_routing(route_tables_warp(p, L, smem, lane, blockIdx.x == 0));
            }
        }
    } else if (cw == 0) {
        publish_routing(load_tables_warp(p, L, smem, lane));
    }
    // shared-expert gate per token (only the shared down items use it; misc[7])
    if (cw == kDkCons - 1) {
        if (p.sh && p.w_sgate) {
            // lane l sums the gate row's 8-value chunks l, l + 32, ... (a few
            // loads in flight; later tokens find the row in L1), then the warp
            // adds the lanes' sums
            const uint4 *wrow = reinterpret_cast<const uint4 *>(p.w_sgate);
#pragma unroll 1
            for (int t = 0; t < T; ++t) {
                float z = 0.f;
#pragma unroll 4
                for (int c = lane; c < H / 8; c += 32) {
                    const uint4 wv = __ldg(wrow + c);
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * xstr + c * 8);
                    const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
                    const __half2 *wh = reinterpret_cast<const __half2 *>(&wv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 a = __half22float2(xh[q]), b = __half22float2(wh[q]);
                        z = fmaf(a.x, b.x, z);
                        z = fmaf(a.y, b.y, z);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                if (lane == 0) gamma[t] = 1.0f / (1.0f + expf(-z));
            }
        } else if (lane < T) {
            gamma[lane] = 1.0f;
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            *reinterpret_cast<volatile int *>(misc + 7) = 1;
        }
    }

    // Counts a gate/up item into its column block; the warp that completes the
    // block finalizes it, frees the slot, and publishes h to the down items.
    auto gu_done = [&](const DHeader &h, int nk, uint2 *hf, size_t hf_kstride, int *rdy, int amount) {
        __syncwarp();
        int old = 0;
        if (lane == 0) {
            __threadfence_block();  // this warp's slot sums before the count
            old = atomicAdd(scnt + h.slot, 1);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != h.nitems - 1) return;
        __threadfence_block();  // every item's slot sums are visible past the count
        finalize_block(sacc + (size_t)h.slot * L.slot_floats, T, nk, lane, hf, hf_kstride);
        __syncwarp();
        if (lane == 0) {
            scnt[h.slot] = 0;
            __threadfence_block();
            sfree[h.slot] = h.bseq + nst;  // the slot's next block
        }
        __threadfence();  // this lane's h fragments before the ready count
        __syncwarp();
        if (lane == 0) atomicAdd(rdy, amount);
    };

    constexpr int NTW = 2 * MS;  // INT4 gate+up tiles per k-step
    constexpr int KB = 2 / MS;   // k-steps per 512 B block
    constexpr int BPG = 8 / KB;  // blocks per group
    const int gbytes = 132 * 16 * MS;
    while (true) {
        int idx = 0;
        if (lane == 0) idx = atomicAdd(&misc[2], 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        const int st = idx % nst;
        // Wait for fill number idx of stage st.  Consumers take stages by
        // ticket, so this warp may wait for a stage whose previous fill has not
        // landed yet; a parity wait cannot tell those two phases apart, so the
        // fill is accepted only when its header carries this ticket.
        bool got = false;
        [[maybe_unused]] const unsigned long long twf = TL_NOW();
        {
            const uint32_t par = (uint32_t)(idx / nst) & 1;
            const volatile int *seqp = &hdrs[st].seq;
            const uint64_t t0 = global_timer_ns();
            while (true) {
                // every lane waits on the barrier itself (each needs the
                // completion's ordering); the fill is taken once all have seen
                // it, so the warp leaves the loop together
                const bool seen = mbar_try_wait_sleep(&full[st], par, kDkSleepNs) && *seqp == idx;
                if (__all_sync(0xffffffffu, seen)) {
                    got = true;
                    break;
                }
                if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
                if (__any_sync(0xffffffffu, global_timer_ns() - t0 > p.wait_budget_ns)) {
                    // the state of the ring at the wait that gave up, for diagnosis
                    if (lane == 0 && atomicCAS(&p.hdr->pad[0], 0u, 1u) == 0u) {
                        p.hdr->pad[1] = (uint32_t)idx;
                        p.hdr->pad[2] = (uint32_t)st;
                        p.hdr->pad[3] = (uint32_t)*seqp;
                        p.hdr->pad[4] = (uint32_t)misc[2];
                        p.hdr->pad[5] = (uint32_t)misc[14];
                        p.hdr->pad[6] = (uint32_t)misc[3];
                        p.hdr->pad[7] = blockIdx.x;
                        p.hdr->pad[8] = (uint32_t)nst;
                        p.hdr->pad[9] = mbar_try_wait(&full[st], par) ? 1u : 0u;
                        p.hdr->pad[10] = (uint32_t)hdrs[st].kind;
                        p.hdr->pad[11] = (uint32_t)cw;
                        for (int j = 0; j < nst && j < 16; ++j) p.hdr->pad[12 + j] = (uint32_t)hdrs[j].seq;
                    }
                    record_timeout(&p.hdr->status, SITE_FILL);
                    *abort_flag = 1;
                    break;
                }
            }
        }
        if (!got) break;
        const DHeader h = hdrs[st];
        [[maybe_unused]] const uint32_t tr_got = TR_NOW();
        if (TL_ON && lane == 0) {
            TL_ADD(p.tl_slot, TL_W_FULL, TL_NOW() - twf);
            TL_FIRST(p.tl_slot, TL_FIRST_FILL);
            if (h.kind == DK_SD || h.kind == DK_RD) TL_FIRST(p.tl_slot, TL_DN_W_FIRST);
            if (h.kind == DK_RG) TL_FIRST(p.tl_slot, TL_RG_FIRST);
        }
        const uint8_t *stage = ring + (size_t)st * L.stage;
        if (h.kind == DK_DONE || h.kind == DK_NOP) {
            // release it too: with fewer stages than warps the end markers reuse stages
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (h.kind == DK_DONE) break;
            continue;
        }
        const int *stn = reinterpret_cast<const int *>(smem + L.stn);
        const TokEntry *ste = reinterpret_cast<const TokEntry *>(smem + L.ste);
        const uint2 *hsl = reinterpret_cast<const uint2 *>(stage + L.hs_off);
        if (h.kind == DK_SD || h.kind == DK_RD) {
            // the intermediate slice lands after the weights (poller's copy); the
            // warp goes on only if every lane saw it
            [[maybe_unused]] const unsigned long long twh = TL_NOW();
            const bool hs_ok =
                mbar_wait_sleep_bounded(&hfull[st], (uint32_t)h.hpar, abort_flag, &p.hdr->status, p.wait_budget_ns);
            if (!__all_sync(0xffffffffu, hs_ok)) {
                *abort_flag = 1;
                break;
            }
            if (TL_ON && lane == 0) {
                TL_ADD(p.tl_slot, TL_W_HFULL, TL_NOW() - twh);
                TL_FIRST(p.tl_slot, TL_DN_H_FIRST);
                if (h.kind == DK_RD) TL_LAST(p.tl_slot, TL_RD_H_LAST);
            }
        }
        [[maybe_unused]] const unsigned long long tc = TL_NOW();  // profiling build: item compute start
        [[maybe_unused]] const uint32_t tr_h = TR_NOW();
#if TL_ON
        auto tr_item = [&](int kind) {
            if (TR_ON()) {
                const uint32_t i = atomicAdd(&s_tr.nitem, 1u);
                if (i < (uint32_t)kTrItems) {
                    s_tr.item[i][0] = ((uint32_t)cw << 8) | (uint32_t)kind;
                    s_tr.item[i][1] = tr_got;
                    s_tr.item[i][2] = tr_h;
                    s_tr.item[i][3] = TR_NOW();
                }
            }
        };
#endif
        if (h.kind == DK_SG) {
            // shared gate/up: 16 columns (tiles: gate, up), k-steps [k0, k0+n) of H
            // two accumulator sets (even / odd k-steps) in registers: the k loop
            // is unrolled by two so that no accumulator index is dynamic
            float acc[2][2][4] = {};
            const bool okx = g < T;
            const __half *xr = xs + (okx ? g : 0) * xstr + 2 * q4;
            for (int ks = 0; ks < h.n; ks += 2) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u == 1 && ks + 1 >= h.n) break;
                    const uint32_t b0 = okx ? lds32(xr + 16 * (h.k0 + ks + u)) : 0u;
                    const uint32_t b1 = okx ? lds32(xr + 16 * (h.k0 + ks + u) + 8) : 0u;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint4 v = lds128(stage + ((size_t)(ks + u) * 2 + t) * 512 + lane * 16);
                        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
                        mma_16816(acc[u][t], a, b0, b1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // the stage is read
            float *sa = sacc + (size_t)h.slot * L.slot_floats;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int col = 2 * q4 + hf;
                    if (col < T) {
                        atomicAdd(sa + (size_t)(32 * t + g) * T + col, acc[0][t][hf] + acc[1][t][hf]);
                        atomicAdd(sa + (size_t)(32 * t + g + 8) * T + col, acc[0][t][2 + hf] + acc[1][t][2 + hf]);
                    }
                }
            }
            [[maybe_unused]] const unsigned long long tg = TL_NOW();
            gu_done(h, 1, p.hf_s + (size_t)h.blk * T * 4, 0, p.rdy_s + h.blk / kDkSdSteps, 1);
            if (TL_ON && lane == 0) {
                TL_ADD(p.tl_slot, TL_C_GU_DONE, TL_NOW() - tg);
                TL_ADD(p.tl_slot, TL_C_SG, TL_NOW() - tc);
#if TL_ON
                tr_item(DK_SG);
#endif
                TL_LAST(p.tl_slot, TL_SG_LAST);
                TL_LAST(p.tl_slot, TL_GU_LAST);
                TL_ADD(p.tl_slot, TL_N_SG, 1);
            }
            continue;
        }
        if (h.kind == DK_RG) {
            // routed INT4 (or Q8_0) gate/up: slice of S = 16*MS columns, groups [k0, k0+n) of H
            const int n_e = min(max(stn[h.a], 0), T);
            const bool okx = g < n_e;
            int tok = okx ? ste[h.a * T + g].tok : 0;
            tok = (tok >= 0 && tok < T) ? tok : 0;
            const __half *xr = xs + tok * xstr + 2 * q4;
            float run[NTW][4] = {};
            if constexpr (Q8) {
                gguf_rg_q8<NTW>(run, stage, h.k0, h.n, xr, okx, lane);
            } else if constexpr (Q2K) {
                const __half *sxh = reinterpret_cast<const __half *>(smem + L.sx16) + tok * (H / 16);
                gguf_rg_q2k<NTW>(run, stage, h.k0, h.n, xr, okx, lane, sxh, sxh + T * (H / 16));
            } else if constexpr (Q4K) {
                const __half *sxh = reinterpret_cast<const __half *>(smem + L.sx16) + tok * (H / 32);
                gguf_rg_q4k<NTW>(run, stage, h.k0, h.n, xr, okx, lane, sxh, sxh + T * (H / 32));
            } else {
                // Raw codes into the mma: rows m < 8 of a tile get 1024 + q, rows m >= 8
                // get 1024 + 16 q (the magic-exponent fragments without their fix-up).
                // Starting each group's accumulator at -1032 (resp. -1152) times the
                // group's x sum leaves sum (q - 8) x (resp. 16 times it): the zero
                // point and the x16 fold into the start value and the row scale.
                const int ng = H / 128;
                int tc0 = 2 * q4 < n_e ? ste[h.a * T + 2 * q4].tok : 0;
                int tc1 = 2 * q4 + 1 < n_e ? ste[h.a * T + 2 * q4 + 1].tok : 0;
                tc0 = (tc0 >= 0 && tc0 < T) ? tc0 : 0;
                tc1 = (tc1 >= 0 && tc1 < T) ? tc1 : 0;
                const float *sx0 = sxs + tc0 * ng, *sx1 = sxs + tc1 * ng;
                for (int gr = 0; gr < h.n; ++gr) {
                    const uint8_t *gp = stage + (size_t)gr * gbytes;
                    const __half *scp = reinterpret_cast<const __half *>(gp);
                    const float s0 = sx0[h.k0 + gr], s1 = sx1[h.k0 + gr];
                    float acc[NTW][4];
#pragma unroll
                    for (int t = 0; t < NTW; ++t) {
                        // with zero points z: start at -(1024 + z) and -(1024 + 16 z) times the sum
                        float za = 8.f, zb = 8.f;
                        if constexpr (ZP) {
                            const __half *zp = reinterpret_cast<const __half *>(stage + L.hs_off) + gr * 32 * MS;
                            za = __half2float(zp[t * 16 + g]);
                            zb = __half2float(zp[t * 16 + g + 8]);
                        }
                        const float ca = -(1024.f + za), cb = -(1024.f + 16.f * zb);
                        acc[t][0] = ca * s0;
                        acc[t][1] = ca * s1;
                        acc[t][2] = cb * s0;
                        acc[t][3] = cb * s1;
                    }
#pragma unroll
                    for (int ib = 0; ib < BPG; ++ib) {
                        const uint4 v = lds128(gp + 64 * MS + ib * 512 + lane * 16);
                        const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int ki = 0; ki < KB; ++ki) {
                            const int ks = (h.k0 + gr) * 8 + ib * KB + ki;
                            const uint32_t b0 = okx ? lds32(xr + 16 * ks) : 0u;
                            const uint32_t b1 = okx ? lds32(xr + 16 * ks + 8) : 0u;
#pragma unroll
                            for (int t = 0; t < NTW; ++t) {
                                uint32_t a[4];
                                codes_frag(words[ki * NTW + t], a);
                                mma_16816(acc[t], a, b0, b1);
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < NTW; ++t) {
                        const float sa = __half2float(scp[t * 16 + g]);
                        const float sb = __half2float(scp[t * 16 + g + 8]) * 0.0625f;
                        run[t][0] = fmaf(sa, acc[t][0], run[t][0]);
                        run[t][1] = fmaf(sa, acc[t][1], run[t][1]);
                        run[t][2] = fmaf(sb, acc[t][2], run[t][2]);
                        run[t][3] = fmaf(sb, acc[t][3], run[t][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // the stage is read
            float *sa = sacc + (size_t)h.slot * L.slot_floats;
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                const int row = 32 * (t < MS ? 0 : 1) + 16 * (t % MS) + g;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int col = 2 * q4 + hf;
                    if (col < n_e) {
                        atomicAdd(sa + (size_t)row * T + col, run[t][hf]);
                        atomicAdd(sa + (size_t)(row + 8) * T + col, run[t][2 + hf]);
                    }
                }
            }
            [[maybe_unused]] const unsigned long long tg = TL_NOW();
            gu_done(h, MS, p.hf_r + ((size_t)h.a * (I / 16) + (size_t)h.blk * MS) * T * 4, (size_t)T * 4,
                    p.rdy_r + h.a * geo.rd_nr + (h.blk * 16 * MS / 128) / geo.rd_gpi, MS);
            if (TL_ON && lane == 0) {
                TL_ADD(p.tl_slot, TL_C_GU_DONE, TL_NOW() - tg);
                TL_ADD(p.tl_slot, TL_C_RG, TL_NOW() - tc);
#if TL_ON
                tr_item(DK_RG);
#endif
                TL_LAST(p.tl_slot, TL_RG_LAST);
                TL_LAST(p.tl_slot, TL_GU_LAST);
                TL_ADD(p.tl_slot, TL_N_RG, 1);
            }
            continue;
        }
        if (h.kind == DK_SD) {
            // shared down: output pair blk (32 outputs), k-steps [k0, k0+n) of I_s
            float acc[2][2][4] = {};  // even / odd k-steps, as in the gate/up items
            const bool okb = g < T;
            for (int ks = 0; ks < h.n; ks += 2) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u == 1 && ks + 1 >= h.n) break;
                    uint2 bv = make_uint2(0u, 0u);
                    if (okb) bv = *reinterpret_cast<const uint2 *>(hsl + ((size_t)(ks + u) * T + g) * 4 + q4);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 v = lds128(stage + ((size_t)(ks + u) * 2 + q) * 512 + lane * 16);
                        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
                        mma_16816(acc[u][q], a, bv.x, bv.y);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // the stage is read
            if (p.mode != 0 && !*reinterpret_cast<volatile int *>(misc + 7)) {  // the gate (set early on)
                const uint64_t t0 = global_timer_ns();
                while (!*reinterpret_cast<volatile int *>(misc + 7) && !*abort_flag) {
                    if (global_timer_ns() - t0 > p.wait_budget_ns) {
                        record_timeout(&p.hdr->status, SITE_GATE);
                        *abort_flag = 1;
                    }
                }
                __threadfence_block();
            }
            const int n0 = 32 * h.blk + 4 * g;
            [[maybe_unused]] const unsigned long long to = TL_NOW();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int col = 2 * q4 + hf;
                if (col < T) {
                    const float w = p.mode == 0 ? 1.f : gamma[col];
                    float4 o;
                    o.x = (acc[0][0][hf] + acc[1][0][hf]) * w;
                    o.y = (acc[0][0][2 + hf] + acc[1][0][2 + hf]) * w;
                    o.z = (acc[0][1][hf] + acc[1][1][hf]) * w;
                    o.w = (acc[0][1][2 + hf] + acc[1][1][2 + hf]) * w;
                    atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)col * H + n0), o);
                }
            }
            if (TL_ON && lane == 0) {
                TL_ADD(p.tl_slot, TL_C_OUT, TL_NOW() - to);
                TL_ADD(p.tl_slot, TL_C_SD, TL_NOW() - tc);
#if TL_ON
                tr_item(DK_SD);
#endif
                TL_LAST(p.tl_slot, TL_SD_LAST);
                TL_LAST(p.tl_slot, TL_DN_LAST);
                TL_ADD(p.tl_slot, TL_N_SD, 1);
            }
            continue;
        }
        // DK_RD: routed INT4 (or Q8_0) down: output pair blk, groups [k0, k0+n) of I
        {
            const int n_e = min(max(stn[h.a], 0), T);
            const bool okb = g < n_e;
            float run[2][4] = {};
            if constexpr (Q8DN) {
                gguf_rd_q8(run, stage, h.n, hsl, T, okb, lane);
            } else {
                for (int gr = 0; gr < h.n; ++gr) {
                    const uint8_t *gp = stage + (size_t)gr * kW4ColGroupBytes;
                    const __half *scp = reinterpret_cast<const __half *>(gp);
                    float acc[2][4] = {};
                    float hsum = 0.f;  // zero points: this lane's part of the group's h sum for token g
#pragma unroll
                    for (int ib = 0; ib < 4; ++ib) {
                        const uint4 v = lds128(gp + 64 + ib * 512 + lane * 16);
                        const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int ki = 0; ki < 2; ++ki) {
                            const int ksr = gr * 8 + ib * 2 + ki;  // k-step within the slice
                            uint2 bv = make_uint2(0u, 0u);
                            if (okb) bv = *reinterpret_cast<const uint2 *>(hsl + ((size_t)ksr * T + g) * 4 + q4);
                            if constexpr (ZP) {
                                const float2 f0 = __half22float2(u32_as_h2(bv.x)), f1 = __half22float2(u32_as_h2(bv.y));
                                hsum += (f0.x + f0.y) + (f1.x + f1.y);
                            }
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                uint32_t a[4];
                                dequant_frag(words[ki * 2 + q], a);
                                mma_16816(acc[q], a, bv.x, bv.y);
                            }
                        }
                    }
                    if constexpr (ZP) {
                        // (q - z) = (q - 8) + (8 - z): add (8 - z) times the group's h sum of each token
                        hsum += __shfl_xor_sync(0xffffffffu, hsum, 1);
                        hsum += __shfl_xor_sync(0xffffffffu, hsum, 2);
                        const float hc0 = __shfl_sync(0xffffffffu, hsum, 8 * q4);
                        const float hc1 = __shfl_sync(0xffffffffu, hsum, 8 * q4 + 4);
                        const __half *zp = reinterpret_cast<const __half *>(stage + kDkRdZeroOff) + gr * 32;
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float da = 8.f - __half2float(zp[q * 16 + g]);
                            const float db = 8.f - __half2float(zp[q * 16 + g + 8]);
                            acc[q][0] = fmaf(da, hc0, acc[q][0]);
                            acc[q][1] = fmaf(da, hc1, acc[q][1]);
                            acc[q][2] = fmaf(db, hc0, acc[q][2]);
                            acc[q][3] = fmaf(db, hc1, acc[q][3]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float sa = __half2float(scp[q * 16 + g]), sb = __half2float(scp[q * 16 + g + 8]);
                        run[q][0] = fmaf(sa, acc[q][0], run[q][0]);
                        run[q][1] = fmaf(sa, acc[q][1], run[q][1]);
                        run[q][2] = fmaf(sb, acc[q][2], run[q][2]);
                        run[q][3] = fmaf(sb, acc[q][3], run[q][3]);
                    }
                }
            }
            int row[2] = {-1, -1};
            float w[2] = {0.f, 0.f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int col = 2 * q4 + hf;
                if (col < n_e) {
                    row[hf] = ste[h.a * T + col].row;
                    w[hf] = ste[h.a * T + col].scale;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // the stage is read
            const int n0 = 32 * h.blk + 4 * g;
            const int rmax = p.mode == 0 ? T * p.k : T;
            [[maybe_unused]] const unsigned long long to = TL_NOW();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                if (row[hf] >= 0 && row[hf] < rmax) {
                    float4 o;
                    o.x = run[0][hf] * w[hf];
                    o.y = run[0][2 + hf] * w[hf];
                    o.z = run[1][hf] * w[hf];
                    o.w = run[1][2 + hf] * w[hf];
                    atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)row[hf] * H + n0), o);
                }
            }
            if (TL_ON && lane == 0) {
                TL_ADD(p.tl_slot, TL_C_OUT, TL_NOW() - to);
                TL_ADD(p.tl_slot, TL_C_RD, TL_NOW() - tc);
#if TL_ON
                tr_item(DK_RD);
#endif
                TL_LAST(p.tl_slot, TL_DN_LAST);
                TL_ADD(p.tl_slot, TL_N_RD, 1);
            }
        }
    }

    // completion ticket; the last block writes the fp16 output and resets
    __threadfence();  // this thread's output additions, before the block counts as done
    all_sync();
    if (ctid == 0) TLB_FIRST(p.tl_slot, TL_CONS_DONE);
    if (ctid == 0) {
        __threadfence();
        const uint32_t t = atomicAdd(&p.hdr->done_ticket, 1u);
        misc[1] = (t == gridDim.x - 1);
    }
    all_sync();
    if (misc[1]) {
        __threadfence();
        if (p.mode == 2) {
            // batches of 8 float4 per thread, all loads of a batch in flight
            const int n4 = T * H / 4;
            constexpr int kNth = kDkCons * 32, kBatch = 8;
            float4 *acc4 = reinterpret_cast<float4 *>(p.yout);
            for (int i0 = ctid; i0 < n4; i0 += kNth * kBatch) {
                float4 v[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = i0 + j * kNth;
                    v[j] = idx < n4 ? __ldcg(acc4 + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = i0 + j * kNth;
                    if (idx < n4) {
                        uint2 o;
                        o.x = h2_as_u32(__floats2half2_rn(v[j].x, v[j].y));
                        o.y = h2_as_u32(__floats2half2_rn(v[j].z, v[j].w));
                        reinterpret_cast<uint2 *>(p.out)[idx] = o;
                        __stcg(acc4 + idx, make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                }
            }
        }
        for (int i = ctid; i < geo.sd_nr; i += kDkCons * 32) p.rdy_s[i] = 0;
        for (int i = ctid; i < p.nact_max * geo.rd_nr; i += kDkCons * 32) p.rdy_r[i] = 0;
        if (ctid < kDkShards) p.qctr[64 * ctid] = 0;
        if (ctid == 0) p.hdr->done_ticket = 0;
        // no fence here: nothing in this launch reads these words again, and
        // the launch that follows reads them only after this one has completed
        if (ctid == 0) TLB_LAST(p.tl_slot, TL_OUT_DONE);
    }
    if (ctid == 0) TLB_LAST(p.tl_slot, TL_EXIT);
    if (TL_ON) {
        __syncwarp();
        all_sync();
        TL_FLUSH(p.tl_slot, ctid);
    }
}

// ------------------------------------------------------------ launching --
#if TL_ON
static std::atomic<int> g_tl_next{0};
#endif

// The launch's template instances, indexed as launch_draft picks them.
using DraftKernel = void (*)(const DkParams);
static DraftKernel draft_instance(int ki) {
    switch (ki) {
    case 0: return draft_kernel<1, DK_FMT_W4>;
    case 1: return draft_kernel<1, DK_FMT_W4Z>;
    case 2: return draft_kernel<2, DK_FMT_W4>;
    case 3: return draft_kernel<2, DK_FMT_W4Z>;
    case 4: return draft_kernel<1, DK_FMT_Q8>;
    case 5: return draft_kernel<1, DK_FMT_Q2K>;
    case 6: return draft_kernel<1, DK_FMT_Q4K>;
    default: return nullptr;
    }
}
constexpr int kDraftInstances = 7;

// Loads instance ki on the current device and raises its dynamic shared-memory
// limit, once per device.
static int configure_draft(int ki) {
    static int configured[kDraftInstances][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPX_ERR_CUDA;
    if (ki < 0 || ki >= kDraftInstances) return SPX_ERR_UNSUPPORTED;
    if (!configured[ki][dev]) {
        cudaError_t err =
            cudaFuncSetAttribute(draft_instance(ki), cudaFuncAttributeMaxDynamicSharedMemorySize, kDkSmemLimit);
        if (err != cudaSuccess) return record_launch(err);
        configured[ki][dev] = 1;
    }
    return SPX_OK;
}

int draft_preload() {
    for (int ki = 0; ki < kDraftInstances; ++ki) {
        const int st = configure_draft(ki);
        if (st) return st;
    }
    return SPX_OK;
}

size_t draft_scratch_end(size_t base, int T, int H, int I, int I_s, int nact_max) {
    return dk_scratch(base, T, H, I, I_s, nact_max).end;
}

bool draft_supported(int T, int H, int I, int S, int I_s, int E, int k, bool kq) {
    if (kq && (H % 256 || S != 16)) return false;
    if (T < 1 || T > kDraftLaunchMaxT || H % 128 || I % 128 || (S != 16 && S != 32)) return false;
    if (I_s % 16 || E < 1 || k < 1 || E > kMaxE || T * k > kMaxSlots) return false;
    return dk_layout(T, H, 4, k, E < T * k ? E : T * k, E, kq).total <= kDkSmemLimit;
}

int launch_draft(const EngineParams &e, const DraftRouting *rt, size_t ws_scratch_base, bool pdl, cudaStream_t s) {
    DkParams p{};
    p.w4 = e.routed;
    const bool zp = e.w4_zeros != nullptr;
    p.fmt = e.routed_fmt == kFmtQ8    ? DK_FMT_Q8
            : e.routed_fmt == kFmtQ2K ? DK_FMT_Q2K
            : e.routed_fmt == kFmtQ4K ? DK_FMT_Q4K
            : zp                      ? DK_FMT_W4Z
                                      : DK_FMT_W4;
    const bool kq = dk_kquant(p.fmt);
    if (e.w4_zeros) {
        p.zeros_gu = reinterpret_cast<const __half *>(e.w4_zeros);
        p.zeros_dn = reinterpret_cast<const __half *>(e.w4_zeros + w4_zeros_gu_bytes(e.E, e.H, e.I, e.S));
    }
    p.S = e.S;
    p.w4_colblk = p.fmt == DK_FMT_Q8    ? q8_units_bytes(e.E, e.H, e.I)
                  : p.fmt == DK_FMT_Q2K ? q2k_units_bytes(e.E, e.H, e.I)
                  : p.fmt == DK_FMT_Q4K ? q4k_units_bytes(e.E, e.H, e.I)
                                        : w4_colblk_offset(e.E, e.H, e.I, e.S);
    p.sh = e.shared;
    p.w_sgate = e.w_sgate;
    p.I_s = e.shared ? e.I_s : 0;
    p.E = e.E;
    p.I = e.I;
    p.k = e.k;
    p.T = e.T;
    p.H = e.H;
    p.active = e.active;
    p.n_active = e.n_active;
    p.tables = e.tables;
    p.x = e.x;
    p.mode = e.mode;
    p.yout = e.yout;
    p.out = e.out;
    p.hdr = e.hdr;
    p.wait_budget_ns = e.wait_budget_ns;
#if TL_ON
    p.tl_slot = g_tl_next.fetch_add(1) % kTlSlots;
#endif
    p.nact_max = e.E < e.T * e.k ? e.E : e.T * e.k;
    if (rt) {
        p.logits = rt->logits;
        p.renorm = rt->renorm;
        p.topk_ids = rt->topk_ids;
        p.topk_w = rt->topk_w;
        p.elb = rt->elb;
        p.layer = rt->layer;
        p.counts = rt->counts;
        p.offsets = rt->offsets;
        p.sorted_slots = rt->sorted_slots;
        p.active_out = rt->active;
        p.n_active_out = rt->n_active;
    }
    uint8_t *ws = reinterpret_cast<uint8_t *>(e.hdr);
    const DkScratch sc = dk_scratch(ws_scratch_base, e.T, e.H, e.I, p.I_s, p.nact_max);
    p.qctr = reinterpret_cast<uint32_t *>(ws + sc.qctr);
    p.hf_s = reinterpret_cast<uint2 *>(ws + sc.hf_s);
    p.hf_r = reinterpret_cast<uint2 *>(ws + sc.hf_r);
    p.rdy_s = reinterpret_cast<int *>(ws + sc.rdy_s);
    p.rdy_r = reinterpret_cast<int *>(ws + sc.rdy_r);
    int nst = 12;  // <= kDkMaxStages
    DkLayout L = dk_layout(e.T, e.H, nst, e.k, p.nact_max, e.E, kq);
    while (nst > 4 && L.total > kDkSmemLimit) L = dk_layout(e.T, e.H, --nst, e.k, p.nact_max, e.E, kq);
    if (L.total > kDkSmemLimit) return SPX_ERR_UNSUPPORTED;
    p.nstages = nst;
    const int sms = device_sm_count();
    if (sms <= 0) return SPX_ERR_CUDA;
    const int ms = e.S / 16;
    const bool gguf = p.fmt == DK_FMT_Q8 || kq;
    if (gguf && (ms != 1 || zp)) return SPX_ERR_UNSUPPORTED;
    if (kq && e.H % 256) return SPX_ERR_UNSUPPORTED;
    const int ki = p.fmt == DK_FMT_Q8    ? 4
                   : p.fmt == DK_FMT_Q2K ? 5
                   : p.fmt == DK_FMT_Q4K ? 6
                                         : (ms - 1) * 2 + (zp ? 1 : 0);
    const int cst = configure_draft(ki);
    if (cst) return cst;
    const DraftKernel kern = draft_instance(ki);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kDkThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, p);
    return record_launch(err);
}

}  // namespace spx

#if TL_ON
// Profiling build only: clear every slot of phase marks (the next draft launch
// writes slot 0), and copy them out ([kTlSlots][kTlBlocks][kTlEvents] words).
extern "C" __attribute__((visibility("default"))) int spx_timeline_reset(void) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, spx::g_tl) != cudaSuccess) return SPX_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(spx::g_tl)) != cudaSuccess) return SPX_ERR_CUDA;
    if (cudaGetSymbolAddress(&p, spx::g_tr) != cudaSuccess) return SPX_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(spx::g_tr)) != cudaSuccess) return SPX_ERR_CUDA;
    spx::g_tl_next.store(0);
    return SPX_OK;
}
extern "C" __attribute__((visibility("default"))) int spx_timeline_trace(void *host, size_t bytes) {
    if (!host || bytes < sizeof(spx::g_tr)) return SPX_ERR_INVALID_ARG;
    return cudaMemcpyFromSymbol(host, spx::g_tr, sizeof(spx::g_tr)) == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}
extern "C" __attribute__((visibility("default"))) int spx_timeline_read(unsigned long long *host, size_t words) {
    if (!host || words < sizeof(spx::g_tl) / 8) return SPX_ERR_INVALID_ARG;
    return cudaMemcpyFromSymbol(host, spx::g_tl, sizeof(spx::g_tl)) == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}
#endif
