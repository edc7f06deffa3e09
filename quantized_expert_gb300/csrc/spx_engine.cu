// spx_engine.cu -- the expert MLP launch shared by the INT4 draft path, the
// FP16 verify path, the shared expert and the composite layer.
//
// Method (ai.info summary of the Specter paper, Key Contributions 4 and
// "Methodology in Plain English"; richland.au post, "What shipped"):
//  - draft: all active experts' INT4 (GPTQ, group 128) MLPs in ONE launch,
//    dequantised in registers and multiplied with fp16 activations (W4A16);
//  - verify: tokens routed to the same expert are packed together so that each
//    expert's FP16 weights are read once and multiplied by all of its tokens
//    as one dense tensor-core product (the "expert-wise reordering");
//  - the FP16 shared expert runs in the same launch; it does not depend on
//    routing, so it is queued first.
//
// GB300 design.  Persistent grid, one block per SM, each block = 8 consumer
// warps + 1 producer warp.  The consumer warps form one or two groups; each
// group has its own ring of stages and processes its own units, so one group's
// gate/up -> down boundary (cross-warp reduction, SiLU) overlaps the other
// group's streaming.  Work is a dynamic queue of "units": one unit = one
// expert's slice of intermediate columns (an INT4 slice of S columns, or two
// adjacent 16-column FP16 slices), so the gate/up reduction over H and the
// SiLU stay inside one block, and the down projection's partial sums over
// units are added into fp32 outputs with vector atomics (no grid-wide
// barrier; only the last 16 blocks to finish wait for the rest, to share the
// fp16 output pass).  A unit is contiguous in HBM
// (repacked once at load time: mma fragment order, GPTQ group scales in front
// of each group's codes) and is streamed by the producer with bulk copies
// (TMA engine) into a ring of shared-memory stages guarded by mbarriers.
// The unit's expert id and slice travel in the stage header and its token
// table is bulk-copied next to the first chunk, so consumers never wait on a
// global load.  Consumers keep partial sums in registers for the whole
// gate/up phase of a slice and reduce across warps once per slice with
// shared-memory atomics.
#include "spx_internal.cuh"

#include <limits.h>
#include <math.h>

namespace spx {

enum : int { HK_GU = 1, HK_DOWN = 2, HK_DONE = 3 };
// HF_GU_LAST: last gate/up chunk of a (sub-)unit, whose partial sums are then
// reduced; HF_GU_FINAL: last gate/up chunk of the unit (h is computed);
// HF_SUB1: gate/up chunk of the second 16-column slice of an FP16 pair;
// HF_PAIR: the unit is an FP16 pair (a down chunk holds both slices' blocks).
enum : int { HF_UNIT_START = 1, HF_GU_LAST = 2, HF_GU_FINAL = 4, HF_SUB1 = 8, HF_PAIR = 16 };
enum : int { MODE_SORTED = 0, MODE_ACC = 1, MODE_LAYER = 2 };
enum : int { FMT_W4 = 0, FMT_F16 = 1, FMT_W4Z = kFmtW4Z };  // FMT_W4Z: INT4 with per-group zero points

struct __align__(16) ChunkHeader {
    int unit;
    int kind;
    int b0;      // first block (INT4 gate/up: group) of the chunk within its section
    int nb;      // blocks in the chunk
    int flags;
    int e;       // expert (routed units)
    int i0;      // first intermediate column of the slice
    int shared;  // 1: shared-expert unit
};

constexpr int kMetaBytes = 1152;                  // >= kTableBytes, multiple of 128
// A stage holds one chunk of weights (a multiple of 1 KB chosen per launch,
// see choose_geometry) followed by the token table area.
static_assert(kTableBytes <= (size_t)kMetaBytes, "table fits the stage meta area");
// The meta area a launch needs: the table header and T entries, in 128-byte units.
__host__ __device__ inline int meta_bytes_for(int T) { return (16 + 16 * T + 127) & ~127; }
constexpr int kHsStride = 40;                     // halves per intermediate row (32 + 8 pad)
constexpr int kEpiBlocks = 16;                    // blocks sharing the fp16 output pass

struct SmemLayout {
    int bars, hdrs, gamma, misc, red, hs, sd, zd, xsum, xs, ring, total;
    int xs_stride;  // halves per activation row
    int red_rs;     // floats per red row
};

// Widest unit a launch reduces: the INT4 slice width, at least an FP16 pair.
__host__ __device__ inline int engine_smax(bool w4, int S) { return w4 && S > 2 * kF16S ? S : 2 * kF16S; }

// G groups of 8/G consumer warps; nsg stages per group.
// red: per group, [2*smax][T] fp32 gate/up sums (the group's warps add into it);
// hs : per group, [npad][kHsStride] fp16 intermediate; sd: per group, 2 x [H]
// fp16 down-scale rows (INT4 only, double-buffered by unit parity); with zero
// points (zp) zd: the same for the down zero-point rows, and xsum: [T][H/128]
// fp32 sums of each activation row over each group of 128; with GGUF K-quant
// gate/up (kqs = 16 for Q2_K, 32 for Q4_K) xsum holds each row's sums over
// kqs rows as fp16 pairs: [T][H/kqs] hi, then [T][H/kqs] lo.
__host__ __device__ inline SmemLayout smem_layout(int T, int H, int npad, int smax, bool w4, int G, int nsg,
                                                  int chunk, bool zp = false, int kqs = 0) {
    SmemLayout L;
    const int nst = G * nsg;
    int o = 0;
    L.bars = o;
    o += (2 * nst + G + 2) * 8;  // full, empty, group, all-consumer, activation barriers
    o = (o + 15) & ~15;
    L.hdrs = o;
    o += nst * (int)sizeof(ChunkHeader);
    L.gamma = o;
    o += kMaxT * 4;
    L.misc = o;
    o += 64;
    L.red = o;
    L.red_rs = T;  // token columns past T are never written
    o += G * 2 * smax * T * 4;
    L.hs = o;
    o += G * npad * kHsStride * 2;
    o = (o + 15) & ~15;
    L.sd = o;
    if (w4) o += G * 2 * H * 2;
    o = (o + 15) & ~15;
    L.zd = o;
    if (zp) o += G * 2 * H * 2;
    L.xsum = o;
    if (zp) o += T * (H / 128) * 4;
    if (kqs) o += T * (H / kqs) * 4;
    o = (o + 15) & ~15;
    L.xs = o;
    L.xs_stride = H + 8;
    o += T * (H + 8) * 2;
    o = (o + 127) & ~127;
    L.ring = o;
    o += nst * (chunk + meta_bytes_for(T));
    L.total = o;
    return L;
}

// ------------------------------------------------------------- producer --
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One lane feeds every group's ring.  Each group has its own unit stream:
// units come from the block's share of the global dynamic queue (one unit is
// dequeued ahead per group so its latency overlaps the copies), and chunks are
// issued into whichever group's ring has a free stage.
struct Stream {
    int u, e, fmt, phase, b, nsub, i0;
    int next_u, next_e, pend_u;
    uint32_t it;
    bool done;
    const uint8_t *base;
    const uint8_t *dbase;  // GGUF: the unit's down codes (unit order)
};

// G (groups) is a template parameter so that the per-group stream state
// stays in registers (a loop over a runtime count would index it in memory).
template <int G>
__device__ void producer_loop(const EngineParams &p, uint8_t *smem, const SmemLayout &L, int nsg) {
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + G * nsg;
    ChunkHeader *hdrs = reinterpret_cast<ChunkHeader *>(smem + L.hdrs);
    uint8_t *ring = smem + L.ring;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc);
    const uint64_t pol = policy_evict_first();
    // The activations, the routing and the workspace may all come from the
    // launch this one follows (which may itself have started early): wait
    // for it before anything else.  The consumers touch global memory only
    // after the activation rows, which are copied after this wait.
    griddep_wait();
    {
        // the activation rows [T][H] -> shared rows of H + 8 halves, ahead of
        // the weights (every block reads them: kept in L2)
        uint64_t *xbar = full + 2 * G * nsg + G + 1;
        const uint64_t keep = policy_evict_last();
        mbar_arrive_expect_tx(xbar, (uint32_t)(p.T * p.H * 2));
        for (int t = 0; t < p.T; ++t)
            bulk_g2s(smem + L.xs + (size_t)t * L.xs_stride * 2, p.x + (size_t)t * p.H, (uint32_t)(p.H * 2), xbar, keep);
    }
    // FP16 units are pairs of adjacent 16-column slices (the last slice alone
    // when the count is odd): the pair's down chunks hold both slices'
    // blocks, so each output partial sum covers 32 intermediate columns and
    // the fp32 output atomics halve.  Shared units are queued first.
    const int nu_sh = p.shared ? p.I_s / kF16S : 0;
    const int n_sh = (nu_sh + 1) / 2;
    const int H = p.H;
    const bool rf16 = p.routed_fmt == FMT_F16;
    const int nu_r = p.I / p.S;                      // routed slices per expert
    const int spe = rf16 ? (nu_r + 1) / 2 : nu_r;    // routed units per expert
    int n_total = -1;

    auto total_units = [&]() -> int {
        if (n_total < 0) {
            int nr = 0;
            if (p.routed_enabled) {
                griddep_wait();  // routing results of the preceding launch
                int na = __ldcg(p.n_active);
                na = na < 0 ? 0 : (na > p.E ? p.E : na);
                nr = na * spe;
            }
            n_total = n_sh + nr;
        }
        return n_total;
    };
    // routed queue index -> active-expert index, first slice, slices
    auto routed_slot = [&](int ur, int &a, int &i, int &nsub) {
        a = ur / spe;
        const int j = ur - a * spe;
        i = rf16 ? 2 * j : j;
        nsub = rf16 && i + 1 < nu_r ? 2 : 1;
    };
    // Queue: stream g of block b starts with unit b*G + g; later units come
    // from the counter (offset by the stream count).  Each stream keeps two
    // units ahead: the next one, whose expert id load was issued a unit
    // earlier, and a counter value fetched a unit earlier, so the producer
    // never waits on a queue round trip while streams are running.
    const int nstreams = (int)gridDim.x * G;
    auto fetch = [&]() -> int { return (int)atomicAdd(&p.hdr->work_counter, 1u) + nstreams; };
    // expert id of unit u (routed units; the load is issued, not waited for)
    auto resolve = [&](int u, int &e) {
        e = -1;
        if (u >= n_sh && p.routed_enabled) {
            int a, i, ns;
            routed_slot(u - n_sh, a, i, ns);
            if (a < p.E) {
                griddep_wait();  // routing results of the preceding launch
                e = __ldcg((p.order ? p.order : p.active) + a);
            }
        }
    };
    // Cache-aware calls: expert e's weights may be read once ready[e] is set
    // (bounded wait; on expiry the status word records SPX_ERR_TIMEOUT and the
    // block stops).  The acquire orders the flag before the weights, the proxy
    // fence before the bulk copies that read them.
    auto ready_wait = [&](int e) -> bool {
        if (ld_acquire_u32(p.ready + e) == 0u) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_u32(p.ready + e) == 0u) {
                if (*abort_flag || global_timer_ns() - t0 > p.wait_budget_ns) {
                    record_timeout(&p.hdr->status, SITE_ENGINE);
                    *abort_flag = 1;
                    return false;
                }
                __nanosleep(256);
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        return true;
    };
    auto valid_unit = [&](int u) -> bool { return u >= 0 && (u < n_sh || u < total_units()); };

    Stream s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        s[g].u = -1;
        s[g].it = 0;
        s[g].done = false;
        s[g].next_u = (int)blockIdx.x * G + g;
        resolve(s[g].next_u, s[g].next_e);
        s[g].pend_u = fetch();
    }
    const int chunk = p.chunk;
    // zero points: a gate/up chunk carries its groups' zero points (2S fp16
    // per group, as the scales) after their codes
    const bool zp = p.w4_zeros != nullptr && !rf16;
    const int W4GPC = chunk / ((int)w4_group_bytes(p.S) + (zp ? 4 * p.S : 0));  // whole INT4 groups per chunk
    // GGUF routed experts (S = 16): gate/up in groups of 128 rows (Q8_0) or
    // super-blocks of 256 (Q2_K, Q4_K), down as 512 B pair blocks in unit order
    const bool gg = p.routed_fmt == kFmtQ8 || p.routed_fmt == kFmtQ2K || p.routed_fmt == kFmtQ4K;
    const int gg_gb = p.routed_fmt == kFmtQ8 ? kQ8GroupBytes : p.routed_fmt == kFmtQ2K ? kQ2kSbBytes : kQ4kSbBytes;
    const int gg_ngr = p.routed_fmt == kFmtQ8 ? H / 128 : H / 256;
    const size_t gg_ub = (size_t)gg_ngr * gg_gb;
    const int GGPC = chunk / gg_gb;  // whole GGUF groups per chunk
    long long t_prog = clock64();
    const long long budget = (long long)p.wait_budget_ns * 2;  // cycles at ~2 GHz
    bool aborted = false;
    while (true) {
        bool all_done = true, progressed = false, stop = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            Stream &S_ = s[g];
            if (S_.done) continue;
            all_done = false;
            const int st = g * nsg + (int)(S_.it % nsg);
            if (!mbar_try_wait(&empty[st], ((S_.it / nsg) & 1) ^ 1)) continue;
            ChunkHeader h;
            const uint8_t *src = nullptr;
            uint32_t bytes = 0, meta_bytes = 0;
            const void *meta = nullptr;
            if (S_.u < 0) {
                const int u = S_.next_u, e = S_.next_e;
                if (!valid_unit(u)) {
                    h = ChunkHeader{};
                    h.kind = HK_DONE;
                    hdrs[st] = h;
                    mbar_arrive(&full[st]);
                    S_.it++;
                    S_.done = true;
                    progressed = true;
                    continue;
                }
                S_.next_u = S_.pend_u;
                resolve(S_.next_u, S_.next_e);
                S_.pend_u = fetch();
                if (u >= n_sh && (e < 0 || e >= p.E)) continue;  // unusable routing entry: skip the unit
                if (p.ready && u >= n_sh && !ready_wait(e)) {
                    stop = true;
                    break;
                }
                S_.u = u;
                S_.e = u < n_sh ? 0 : e;
                S_.fmt = u < n_sh ? FMT_F16 : p.routed_fmt;
                S_.phase = 0;
                S_.b = 0;
                if (u < n_sh) {
                    S_.base = p.shared + (size_t)(2 * u) * f16_unit_bytes(H);
                    S_.nsub = 2 * u + 1 < nu_sh ? 2 : 1;
                } else {
                    int a, i;
                    routed_slot(u - n_sh, a, i, S_.nsub);
                    S_.i0 = i * p.S;
                    const size_t uix = (size_t)e * nu_r + i;
                    if (gg) {
                        S_.base = p.routed + uix * gg_ub;
                        S_.dbase = p.routed + gguf_udn_offset(p.E, H, p.I, p.routed_fmt) + uix * ((size_t)H * 16);
                    } else {
                        S_.base = p.routed + uix * (S_.fmt == FMT_W4 ? w4_unit_bytes(H, p.S) : f16_unit_bytes(H));
                    }
                }
            }
            const bool shared = S_.u < n_sh;
            h.unit = S_.u;
            h.shared = shared;
            h.e = S_.e;
            h.i0 = shared ? S_.u * 2 * kF16S : S_.i0;
            h.flags = 0;
            const uint8_t *src2 = nullptr;  // second slice of an FP16 pair's down chunk, or INT4 zero points
            uint32_t bytes2 = 0;
            if (gg && !shared) {
                if (S_.phase == 0) {
                    h.kind = HK_GU;
                    h.b0 = S_.b;
                    h.nb = min(GGPC, gg_ngr - S_.b);
                    h.flags = (S_.b == 0 ? HF_UNIT_START : 0) | (S_.b + h.nb == gg_ngr ? HF_GU_LAST | HF_GU_FINAL : 0);
                    src = S_.base + (size_t)S_.b * gg_gb;
                    bytes = h.nb * (uint32_t)gg_gb;
                    S_.b += h.nb;
                    if (S_.b >= gg_ngr) S_.phase = 1, S_.b = 0;
                } else {
                    const int nbd = H / 32;
                    h.kind = HK_DOWN;
                    h.b0 = S_.b;
                    h.nb = min(chunk / 512, nbd - S_.b);
                    src = S_.dbase + (size_t)S_.b * 512;
                    bytes = h.nb * 512;
                    S_.b += h.nb;
                    if (S_.b >= nbd) S_.u = -1;
                }
            } else if (S_.fmt == FMT_W4) {
                const int S = p.S;
                const int ngr = H / 128;
                const int nbd = (int)(w4_dn_bytes(H, S) / 512);
                if (S_.phase == 0) {
                    h.kind = HK_GU;
                    h.b0 = S_.b;
                    h.nb = min(W4GPC, ngr - S_.b);
                    h.flags = (S_.b == 0 ? HF_UNIT_START : 0) | (S_.b + h.nb == ngr ? HF_GU_LAST | HF_GU_FINAL : 0);
                    src = S_.base + (size_t)S_.b * w4_group_bytes(S);
                    bytes = h.nb * (uint32_t)w4_group_bytes(S);
                    if (zp) {
                        const size_t uix = (size_t)S_.e * nu_r + S_.i0 / S;
                        src2 = p.w4_zeros + (uix * (H / 128) + S_.b) * 4 * S;
                        bytes2 = h.nb * 4u * (uint32_t)S;
                    }
                    S_.b += h.nb;
                    if (S_.b >= ngr) S_.phase = 1, S_.b = 0;
                } else {
                    h.kind = HK_DOWN;
                    h.b0 = S_.b;
                    h.nb = min(chunk / 512, nbd - S_.b);
                    src = S_.base + w4_gu_bytes(H, S) + (size_t)S_.b * 512;
                    bytes = h.nb * 512;
                    S_.b += h.nb;
                    if (S_.b >= nbd) S_.u = -1;
                }
            } else {
                // phase 0 / 1: gate/up of slice 0 / 1; phase 2: down of both
                const int nbg = H / 16, nbd = H / 32;
                const int pair = S_.nsub == 2 ? HF_PAIR : 0;
                if (S_.phase < 2) {
                    const int sub = S_.phase;
                    const bool last = S_.b + min(chunk / 1024, nbg - S_.b) == nbg;
                    h.kind = HK_GU;
                    h.b0 = S_.b;
                    h.nb = min(chunk / 1024, nbg - S_.b);
                    h.flags = (sub == 0 && S_.b == 0 ? HF_UNIT_START : 0) | (last ? HF_GU_LAST : 0) |
                              (last && sub + 1 == S_.nsub ? HF_GU_FINAL : 0) | (sub ? HF_SUB1 : 0) | pair;
                    src = S_.base + (size_t)sub * f16_unit_bytes(H) + (size_t)S_.b * 1024;
                    bytes = h.nb * 1024;
                    S_.b += h.nb;
                    if (S_.b >= nbg) S_.phase = sub + 1 < S_.nsub ? sub + 1 : 2, S_.b = 0;
                } else {
                    h.kind = HK_DOWN;
                    h.b0 = S_.b;
                    h.nb = min(chunk / (1024 * S_.nsub), nbd - S_.b);
                    h.flags = pair;
                    src = S_.base + f16_gu_bytes(H) + (size_t)S_.b * 1024;
                    bytes = h.nb * 1024;
                    if (pair) {
                        src2 = src + f16_unit_bytes(H);
                        bytes2 = bytes;
                    }
                    S_.b += h.nb;
                    if (S_.b >= nbd) S_.u = -1;
                }
            }
            if ((h.flags & HF_UNIT_START) && !shared) {
                meta = p.tables + h.e;
                meta_bytes = (uint32_t)(16 + 16 * p.T);  // table header + up to T entries
            }
            hdrs[st] = h;
            uint8_t *dst = ring + (size_t)st * (chunk + meta_bytes_for(p.T));
            mbar_arrive_expect_tx(&full[st], bytes + bytes2 + meta_bytes);
            bulk_g2s(dst, src, bytes, &full[st], pol);
            if (bytes2) bulk_g2s(dst + bytes, src2, bytes2, &full[st], pol);
            if (meta_bytes) bulk_g2s(dst + chunk, meta, meta_bytes, &full[st], pol);
            S_.it++;
            progressed = true;
        }
        if (stop) {
            aborted = true;
            break;
        }
        if (all_done) break;
        if (progressed) {
            t_prog = clock64();
        } else if (*abort_flag || clock64() - t_prog > budget) {
            record_timeout(&p.hdr->status, SITE_ENGINE);
            *abort_flag = 1;
            aborted = true;
            break;
        }
    }
    // Each stream's counter value fetched ahead may still be in flight: wait
    // for every value (a returned value means the add is done at L2) and
    // fence, so that no add of this block can land after the last block has
    // reset the counter for the next call.
    {
        int seen = 0;
#pragma unroll
        for (int g = 0; g < G; ++g) seen ^= s[g].pend_u;
        if (seen == INT_MIN) atomicCAS(&p.hdr->status, 0, 0);  // reads the values; never true
        __threadfence();
    }
    // Drain: every issued copy has been waited on by the consumers unless the
    // block aborted; in that case wait (bounded) for the copies in flight.
    if (aborted) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint32_t first = s[g].it > (uint32_t)nsg ? s[g].it - nsg : 0;
            for (uint32_t j = first; j < s[g].it; ++j) {
                const int st = g * nsg + (int)(j % nsg);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[st], (j / nsg) & 1) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    }
}

// ------------------------------------------------------------ consumers --
struct Sync {
    uint64_t *bar;
    uint32_t phase;
};

// All warps that share `bar` (initialised with their count) meet here.
__device__ __forceinline__ void group_sync(const EngineParams &p, Sync &sy, volatile int *abort_flag) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(sy.bar);
    mbar_wait_bounded(sy.bar, sy.phase & 1, abort_flag, &p.hdr->status, p.wait_budget_ns);
    sy.phase ^= 1;
    __syncwarp();
}

// RFMT: format of the routed experts (INT4 draft, INT4 with zero points, or
// FP16 verify); the FP16 kernel carries no INT4 code.  Nine warps per block
// put three warps on one SM sub-partition, whose 16K registers cap a thread
// at 168 registers.
//
// Zero points (FMT_W4Z; the AWQ form W = s (q - z), z per group of 128 input
// rows and output column): the mma sums x (q - 8) as for symmetric INT4, and
// the group's term s (8 - z) * (sum of x over the group) is added per token
// column (gate/up); the down projection adds s (8 - z) * (sum of h over the
// unit's S intermediate rows, which lie in one group of 128).
template <int RFMT, int MS4, int NT>
__global__ void __launch_bounds__(kThreads, 1) engine_kernel(const EngineParams p) {
    constexpr bool ZP = RFMT == FMT_W4Z;
    constexpr bool W4R = RFMT == FMT_W4 || ZP;  // INT4 routed experts
    constexpr bool Q2K = RFMT == kFmtQ2K, Q4K = RFMT == kFmtQ4K;
    constexpr bool GG = RFMT == kFmtQ8 || Q2K || Q4K;  // GGUF routed experts (S = 16, Q8_0 down)
    constexpr int KQS = Q2K ? 16 : Q4K ? 32 : 0;       // K-quant gate/up: rows per x sum
    extern __shared__ __align__(128) uint8_t smem[];
    // A launch that follows on the stream may be scheduled as SMs free up; it
    // reads nothing of this one before its own griddepcontrol.wait.
    griddep_launch_dependents();
    const bool has_w4 = (W4R || GG) && p.routed_enabled;  // per-unit down-scale rows
    const int smax = engine_smax(has_w4, p.S);
    const int G = p.groups, nsg = p.nstages;
    const int gwarps = kConsumerWarps / G;
    const SmemLayout L = smem_layout(p.T, p.H, p.npad, smax, has_w4, G, nsg, p.chunk, ZP, KQS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q4 = lane & 3;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + G * nsg;
    uint64_t *gbar = empty + G * nsg;  // one per group
    uint64_t *allbar = gbar + G;       // all consumer warps
    uint64_t *xbar = allbar + 1;       // activation rows landed
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    if (threadIdx.x == 0) {
        for (int s = 0; s < G * nsg; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], gwarps);
        }
        for (int q = 0; q < G; ++q) mbar_init(&gbar[q], gwarps);
        mbar_init(allbar, kConsumerWarps);
        mbar_init(xbar, 1);
        misc[0] = 0;  // abort flag
        misc[1] = 0;  // last-block flag
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            if (G == 2)
                producer_loop<2>(p, smem, L, nsg);
            else
                producer_loop<1>(p, smem, L, nsg);
        }
        return;
    }
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc);
    const int grp_id = warp / gwarps, gw = warp % gwarps;
    const int gtid = gw * 32 + lane;  // thread index within the group
    Sync gs{&gbar[grp_id], 0};
    Sync as{allbar, 0};
    const ChunkHeader *hdrs = reinterpret_cast<const ChunkHeader *>(smem + L.hdrs);
    const uint8_t *ring = smem + L.ring;
    float *gamma = reinterpret_cast<float *>(smem + L.gamma);
    const int xs_stride = L.xs_stride, rs = L.red_rs, npad = p.npad;
    float *red = reinterpret_cast<float *>(smem + L.red) + (size_t)grp_id * 2 * smax * rs;
    __half *hs = reinterpret_cast<__half *>(smem + L.hs) + (size_t)grp_id * npad * kHsStride;
    __half *sdg = reinterpret_cast<__half *>(smem + L.sd) + (size_t)grp_id * 2 * p.H;
    __half *zdg = reinterpret_cast<__half *>(smem + L.zd) + (size_t)grp_id * 2 * p.H;  // ZP only
    const float *xsum = reinterpret_cast<const float *>(smem + L.xsum);                 // ZP only
    const int ngr = p.H / 128;
    __half *xs = reinterpret_cast<__half *>(smem + L.xs);
    const int ctid = threadIdx.x;  // 0..255
    const int H = p.H;

    // zero the groups' gate/up reduction buffers; the activation rows come
    // in by bulk copies the producer issues first
    for (int idx = ctid; idx < G * 2 * smax * rs; idx += kConsumerWarps * 32)
        reinterpret_cast<float *>(smem + L.red)[idx] = 0.f;
    mbar_wait_bounded(xbar, 0, abort_flag, &p.hdr->status, p.wait_budget_ns);
    if (KQS) {  // each activation row's sums over KQS rows, as fp16 pairs hi + lo
        __half *xsh = reinterpret_cast<__half *>(smem + L.xsum);
        const int nsb = p.H / KQS;
        for (int idx = ctid; idx < p.T * nsb; idx += kConsumerWarps * 32) {
            const int t = idx / nsb, b = idx - t * nsb;
            const __half2 *xr2 = reinterpret_cast<const __half2 *>(xs + (size_t)t * L.xs_stride + b * KQS);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < KQS / 2; ++j) {
                const float2 f = __half22float2(xr2[j]);
                sum += f.x + f.y;
            }
            const __half hi = __float2half_rn(sum);
            xsh[idx] = hi;
            xsh[p.T * nsb + idx] = __float2half_rn(sum - __half2float(hi));
        }
    }
    if (ZP) {  // each activation row's sums over the groups of 128
        float *xsw = reinterpret_cast<float *>(smem + L.xsum);
        for (int idx = ctid; idx < p.T * ngr; idx += kConsumerWarps * 32) {
            const int t = idx / ngr, gi = idx - t * ngr;
            const __half2 *xr2 = reinterpret_cast<const __half2 *>(xs + (size_t)t * L.xs_stride + gi * 128);
            float sum = 0.f;
#pragma unroll 8
            for (int j = 0; j < 64; ++j) {
                const float2 f = __half22float2(xr2[j]);
                sum += f.x + f.y;
            }
            xsw[idx] = sum;
        }
    }
    group_sync(p, as, abort_flag);
    // shared-expert gate per token: gamma = 1 / (1 + exp(-x . w_sgate)), else 1
    if (p.shared && p.w_sgate) {
        for (int t = warp; t < p.T; t += kConsumerWarps) {
            float z = 0.f;
            for (int hh = lane * 2; hh < H; hh += 64) {
                const float2 xv = __half22float2(*reinterpret_cast<const __half2 *>(xs + (size_t)t * xs_stride + hh));
                const float2 wv = __half22float2(__ldg(reinterpret_cast<const __half2 *>(p.w_sgate + hh)));
                z = fmaf(xv.x, wv.x, z);
                z = fmaf(xv.y, wv.y, z);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) gamma[t] = 1.0f / (1.0f + expf(-z));
        }
    } else {
        for (int t = ctid; t < p.T; t += kConsumerWarps * 32) gamma[t] = 1.0f;
    }
    group_sync(p, as, abort_flag);

    constexpr int NTW = 2 * MS4;  // INT4 gate+up tiles per k-step (FP16 units use 2)
    constexpr int KH = MS4 > 2 ? MS4 : 2;  // k-steps of the down projection (an FP16 pair has 2)
    // per-warp state of the current unit
    int u_fmt = FMT_F16, u_S = kF16S, u_e = 0, u_i0 = 0, n_e = 0, nact = 0;
    uint32_t ucount = 0;     // units started by this group (selects the down-scale buffer)
    const __half *sdcur = sdg;
    const __half *zdcur = zdg;
    int xoff[NT];
    int ctok[NT][2];     // ZP: tokens of this lane's output columns 2*q4, 2*q4+1 of each n-tile
    float hsum[NT][2];   // ZP: their sums of h over the unit's intermediate rows
    int orow[NT][2];
    float oscl[NT][2];
    float run[NTW][NT][4];                // gate/up partial sums of this warp for the whole unit
    uint32_t hb0[KH][NT], hb1[KH][NT];  // h fragments for the down phase
#pragma unroll
    for (int ks = 0; ks < KH; ++ks)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) hb0[ks][nt] = hb1[ks][nt] = 0u;

    uint32_t it = 0;
    while (it < (1u << 30)) {
        const int st = grp_id * nsg + (int)(it % nsg);
        if (!mbar_wait_bounded(&full[st], (it / nsg) & 1, abort_flag, &p.hdr->status, p.wait_budget_ns)) break;
        const ChunkHeader h = hdrs[st];
        if (h.kind == HK_DONE) break;
        const uint8_t *stage = ring + (size_t)st * (p.chunk + meta_bytes_for(p.T));
        if (h.flags & HF_UNIT_START) {
            // unit setup from the header and the token table in the meta area
            u_fmt = (h.shared || RFMT == FMT_F16) ? FMT_F16 : GG ? RFMT : FMT_W4;
            u_S = u_fmt == FMT_F16 ? kF16S * ((h.flags & HF_PAIR) ? 2 : 1) : p.S;
            u_e = h.e;
            u_i0 = h.i0;
            const TokTable *tb = reinterpret_cast<const TokTable *>(stage + p.chunk);
            int n = h.shared ? p.T : tb->n;
            if (n < 0 || n > p.T || n > 8 * NT) n = 0;
            n_e = n;
            nact = (n + 7) >> 3;
            const int rmax = p.mode == MODE_SORTED ? p.T * p.k : p.T;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int colb = nt * 8 + g;
                int t = -1;
                if (colb < n) {
                    t = h.shared ? colb : tb->e[colb].tok;
                    t = (t >= 0 && t < p.T) ? t : 0;
                }
                xoff[nt] = t < 0 ? -1 : t * xs_stride + 2 * q4;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int col = nt * 8 + 2 * q4 + hf;
                    int r = 0;
                    float sc = 0.f;
                    int ct = 0;
                    if (col < n) {
                        if (h.shared) {
                            r = col;
                            sc = p.mode == MODE_SORTED ? 1.f : gamma[col];
                            ct = col;
                        } else {
                            r = tb->e[col].row;
                            sc = tb->e[col].scale;
                            ct = tb->e[col].tok;
                        }
                    }
                    ctok[nt][hf] = (ct >= 0 && ct < p.T) ? ct : 0;
                    const bool okr = r >= 0 && r < rmax;
                    orow[nt][hf] = okr ? r : 0;
                    oscl[nt][hf] = okr ? sc : 0.f;
                }
            }
#pragma unroll
            for (int t = 0; t < NTW; ++t)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) run[t][nt][r] = 0.f;
            if ((W4R && u_fmt == FMT_W4) || (GG && u_fmt == RFMT)) {
                // fetch this unit's down-scale row into the group's buffer for
                // this unit's parity; waited for at the gate/up -> down boundary
                // (INT4: per group of 128 intermediate rows; GGUF Q8_0: per
                // block of 32)
                __half *dst = sdg + (size_t)(ucount & 1) * H;
                const __half *srow =
                    GG ? reinterpret_cast<const __half *>(p.routed + gguf_uds_offset(p.E, H, p.I, RFMT)) +
                             ((size_t)u_e * (p.I / 32) + u_i0 / 32) * H
                       : p.w4_sdown + ((size_t)u_e * (p.I / 128) + u_i0 / 128) * H;
                for (int idx = gtid; idx < H / 8; idx += gwarps * 32) cp_async16(dst + idx * 8, srow + idx * 8);
                if (ZP) {
                    // and its down zero-point row: [E][H/32][I/128][32], 32 outputs a piece
                    __half *zdst = zdg + (size_t)(ucount & 1) * H;
                    const __half *zdn = reinterpret_cast<const __half *>(
                        p.w4_zeros + w4_zeros_gu_bytes(p.E, H, p.I, p.S));
                    const int nig = p.I / 128, gi = u_i0 / 128;
                    for (int idx = gtid; idx < H / 8; idx += gwarps * 32) {
                        const int blk = idx >> 2;
                        cp_async16(zdst + idx * 8, zdn + (((size_t)u_e * (H / 32) + blk) * nig + gi) * 32 + (idx & 3) * 8);
                    }
                    zdcur = zdst;
                }
                cp_async_commit();
                sdcur = dst;
            }
            ++ucount;
        }
        if (n_e > 0 && h.kind == HK_GU) {
            if (W4R && u_fmt == FMT_W4) {
                // blocks of KB k-steps; 8/KB blocks per group after 4S bytes of scales
                constexpr int KB = 2 / MS4;
                constexpr int BPG = 8 / KB;
                const int gb = 132 * u_S;
                const int nblk = h.nb * BPG;
                const int per = (nblk + gwarps - 1) / gwarps;
                const int bb = gw * per, be = min(bb + per, nblk);
                const __half *zsp = reinterpret_cast<const __half *>(stage + (size_t)h.nb * gb);  // ZP: after the codes
                float acc[NTW][NT][4];
                float sA[NTW], sB[NTW], dA[NTW], dB[NTW];  // scales; ZP: 8 - zero point
                int grp = -1;
                bool zfirst = false;  // ZP: this warp holds the group's first block (the group's
                                      // zero-point term is added once, by that warp)
#pragma unroll
                for (int t = 0; t < NTW; ++t) sA[t] = sB[t] = dA[t] = dB[t] = 0.f;
                // adds the finished group's sums, scaled (ZP: with the group's
                // zero-point term per token column when this warp holds the
                // group's first block; a group's blocks may be split between
                // two warps)
                auto flush = [&]() {
                    float xa[NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
                            xa[nt][hf] = ZP && zfirst ? xsum[ctok[nt][hf] * ngr + h.b0 + grp] : 0.f;
#pragma unroll
                    for (int t = 0; t < NTW; ++t)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            run[t][nt][0] = fmaf(sA[t], ZP ? fmaf(dA[t], xa[nt][0], acc[t][nt][0]) : acc[t][nt][0],
                                                 run[t][nt][0]);
                            run[t][nt][1] = fmaf(sA[t], ZP ? fmaf(dA[t], xa[nt][1], acc[t][nt][1]) : acc[t][nt][1],
                                                 run[t][nt][1]);
                            run[t][nt][2] = fmaf(sB[t], ZP ? fmaf(dB[t], xa[nt][0], acc[t][nt][2]) : acc[t][nt][2],
                                                 run[t][nt][2]);
                            run[t][nt][3] = fmaf(sB[t], ZP ? fmaf(dB[t], xa[nt][1], acc[t][nt][3]) : acc[t][nt][3],
                                                 run[t][nt][3]);
                        }
                };
                for (int bl = bb; bl < be; ++bl) {
                    const int gr = bl / BPG, ib = bl - gr * BPG;
                    const uint8_t *gp = stage + (size_t)gr * gb;
                    if (gr != grp) {
                        if (grp >= 0) flush();
                        grp = gr;
                        zfirst = ib == 0;
                        const __half *scp = reinterpret_cast<const __half *>(gp);
#pragma unroll
                        for (int t = 0; t < NTW; ++t) {
                            sA[t] = __half2float(scp[t * 16 + g]);
                            sB[t] = __half2float(scp[t * 16 + g + 8]);
                            if (ZP) {
                                dA[t] = 8.f - __half2float(zsp[gr * 2 * u_S + t * 16 + g]);
                                dB[t] = 8.f - __half2float(zsp[gr * 2 * u_S + t * 16 + g + 8]);
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int r = 0; r < 4; ++r) acc[t][nt][r] = 0.f;
                        }
                    }
                    const uint4 v = lds128(gp + 4 * u_S + ib * 512 + lane * 16);
                    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int ki = 0; ki < KB; ++ki) {
                        const int ks = (h.b0 + gr) * 8 + ib * KB + ki;  // k-step within H
                        uint32_t bf0[NT], bf1[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const bool okx = xoff[nt] >= 0;
                            const __half *xr = xs + (okx ? xoff[nt] : 0) + 16 * ks;
                            bf0[nt] = okx ? lds32(xr) : 0u;
                            bf1[nt] = okx ? lds32(xr + 8) : 0u;
                        }
#pragma unroll
                        for (int t = 0; t < NTW; ++t) {
                            uint32_t a[4];
                            dequant_frag(words[ki * NTW + t], a);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                if (nt < nact) mma_16816(acc[t][nt], a, bf0[nt], bf1[nt]);
                        }
                    }
                }
                if (grp >= 0) flush();
            } else if ((Q2K || Q4K) && u_fmt == RFMT) {
                // GGUF Q2_K / Q4_K: whole super-blocks of 256 rows per warp (the
                // min term is per super-block).  The fragment holds sc*q, exact in
                // fp16 through one fused multiply-add of the magic value 1024 + q,
                // so one accumulator spans the super-block; the mins enter through
                // one more product, of the rows' sub-block mins with the token's
                // sub-block sums of x (fp16 pairs hi + lo); then d and dmin per row.
                constexpr int SBB = Q2K ? kQ2kSbBytes : kQ4kSbBytes;
                const int nsb = h.nb;
                const int per = (nsb + gwarps - 1) / gwarps;
                const int s0 = gw * per, s1 = min(s0 + per, nsb);
                const __half *xsh = reinterpret_cast<const __half *>(smem + L.xsum);
                const int nxs = H / KQS;  // x sums per activation row
                int xtk[NT];              // token of this lane's B column in each n-tile, -1 if none
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xtk[nt] = xoff[nt] >= 0 ? (xoff[nt] - 2 * q4) / xs_stride : -1;
                const __half2 k1024 = u32_as_h2(0x64006400u), km1024 = u32_as_h2(0xE400E400u);
                for (int gr = s0; gr < s1; ++gr) {
                    const uint8_t *sp = stage + (size_t)gr * SBB;
                    const __half *dd = reinterpret_cast<const __half *>(sp);  // d [32], then dmin [32]
                    const int sbg = h.b0 + gr;                              // super-block of H
                    const uint4 c0 = lds128(sp + (Q2K ? kQ2kScaleOff : kQ4kScaleOff) + g * 32);
                    const uint4 c1 = lds128(sp + (Q2K ? kQ2kScaleOff : kQ4kScaleOff) + g * 32 + 16);
                    const uint32_t scw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    float am[2][NT][4];
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int r = 0; r < 4; ++r) am[t][nt][r] = 0.f;
                    if constexpr (Q2K) {
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            const uint4 v = lds128(sp + kQ2kCodeOff + c * 512 + lane * 16);
                            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const int kl = 4 * c + kk;
                                const int ks = sbg * 16 + kl;
                                uint32_t bf0[NT], bf1[NT];
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    const bool okx = xoff[nt] >= 0;
                                    const __half *xr = xs + (okx ? xoff[nt] : 0) + 16 * ks;
                                    bf0[nt] = okx ? lds32(xr) : 0u;
                                    bf1[nt] = okx ? lds32(xr + 8) : 0u;
                                }
                                // the k-step's four scale nibbles (tile t, row g / g+8), in both halves
                                const uint32_t su = ((scw[kl >> 1] >> (16 * (kl & 1))) & 0xFFFFu) * 0x10001u;
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    const __half2 sa2 =
                                        __hsub2(u32_as_h2(lop3_and_or(su >> (8 * t), 0x000F000Fu, 0x64006400u)), k1024);
                                    const __half2 sb2 = __hsub2(
                                        u32_as_h2(lop3_and_or(su >> (8 * t + 4), 0x000F000Fu, 0x64006400u)), k1024);
                                    const __half2 oa2 = __hmul2(sa2, km1024), ob2 = __hmul2(sb2, km1024);
                                    uint32_t a[4];
#pragma unroll
                                    for (int r = 0; r < 4; ++r) {
                                        const uint32_t raw =
                                            lop3_and_or(words[kk] >> (2 * (4 * t + r)), 0x00030003u, 0x64006400u);
                                        a[r] = h2_as_u32(__hfma2(u32_as_h2(raw), (r & 1) ? sb2 : sa2, (r & 1) ? ob2 : oa2));
                                    }
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt)
                                        if (nt < nact) mma_16816(am[t][nt], a, bf0[nt], bf1[nt]);
                                }
                            }
                        }
                    } else {
                        const uint32_t kExp = 0x64646464u;
#pragma unroll 1
                        for (int c = 0; c < 8; ++c) {
                            const uint4 v = lds128(sp + kQ4kCodeOff + c * 512 + lane * 16);
                            const uint32_t words[4] = {v.x, v.y, v.z, v.w};  // [k-step][tile]
                            __half2 sc2[2][2], of2[2][2];                     // (scale, -1024 scale) of rows g, g+8
#pragma unroll
                            for (int t = 0; t < 2; ++t)
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    const uint32_t sel = (2 * t + j) * 0x0101u + 0x4040u;  // byte 2t+j under 0x64
                                    sc2[t][j] = __hsub2(u32_as_h2(__byte_perm(scw[c], kExp, sel)), k1024);
                                    of2[t][j] = __hmul2(sc2[t][j], km1024);
                                }
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const int ks = sbg * 16 + 2 * c + kk;
                                uint32_t bf0[NT], bf1[NT];
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    const bool okx = xoff[nt] >= 0;
                                    const __half *xr = xs + (okx ? xoff[nt] : 0) + 16 * ks;
                                    bf0[nt] = okx ? lds32(xr) : 0u;
                                    bf1[nt] = okx ? lds32(xr + 8) : 0u;
                                }
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    const uint32_t w = words[2 * kk + t];
                                    uint32_t a[4];
#pragma unroll
                                    for (int r = 0; r < 4; ++r) {
                                        const uint32_t raw = lop3_and_or(w >> (4 * r), 0x000F000Fu, 0x64006400u);
                                        a[r] = h2_as_u32(__hfma2(u32_as_h2(raw), sc2[t][r & 1], of2[t][r & 1]));
                                    }
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt)
                                        if (nt < nact) mma_16816(am[t][nt], a, bf0[nt], bf1[nt]);
                                }
                            }
                        }
                    }
                    // d times the code products, then the same accumulators take
                    // the min products (scaled by dmin and subtracted)
                    float da[2], db[2], ma[2], mb[2];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        da[t] = __half2float(dd[t * 16 + g]);
                        db[t] = __half2float(dd[t * 16 + g + 8]);
                        ma[t] = __half2float(dd[32 + t * 16 + g]);
                        mb[t] = __half2float(dd[32 + t * 16 + g + 8]);
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            run[t][nt][0] = fmaf(da[t], am[t][nt][0], run[t][nt][0]);
                            run[t][nt][1] = fmaf(da[t], am[t][nt][1], run[t][nt][1]);
                            run[t][nt][2] = fmaf(db[t], am[t][nt][2], run[t][nt][2]);
                            run[t][nt][3] = fmaf(db[t], am[t][nt][3], run[t][nt][3]);
#pragma unroll
                            for (int r = 0; r < 4; ++r) am[t][nt][r] = 0.f;
                        }
                    uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const bool okx = xtk[nt] >= 0;
                        const __half *xh = xsh + (okx ? xtk[nt] : 0) * nxs + sbg * (256 / KQS) + 2 * q4;
                        const __half *xl = xh + p.T * nxs;
                        bh0[nt] = okx ? lds32(xh) : 0u;
                        bl0[nt] = okx ? lds32(xl) : 0u;
                        bh1[nt] = okx && Q2K ? lds32(xh + 8) : 0u;  // Q4_K: 8 sub-blocks, k >= 8 zero
                        bl1[nt] = okx && Q2K ? lds32(xl + 8) : 0u;
                    }
                    const uint2 mw = lds64(sp + (Q2K ? kQ2kMinOff : kQ4kMinOff) + lane * 8);
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t w = t == 0 ? mw.x : mw.y;
                        uint32_t a[4];
                        if constexpr (Q2K) {
#pragma unroll
                            for (int r = 0; r < 4; ++r)
                                a[r] = h2_as_u32(
                                    __hsub2(u32_as_h2(lop3_and_or(w >> (4 * r), 0x000F000Fu, 0x64006400u)), k1024));
                        } else {
                            const uint32_t kExp = 0x64646464u;
                            a[0] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, kExp, 0x4140u)), k1024));
                            a[1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, kExp, 0x4342u)), k1024));
                            a[2] = 0u;
                            a[3] = 0u;
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nact) {
                                mma_16816(am[t][nt], a, bh0[nt], bh1[nt]);
                                mma_16816(am[t][nt], a, bl0[nt], bl1[nt]);
                            }
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            run[t][nt][0] = fmaf(-ma[t], am[t][nt][0], run[t][nt][0]);
                            run[t][nt][1] = fmaf(-ma[t], am[t][nt][1], run[t][nt][1]);
                            run[t][nt][2] = fmaf(-mb[t], am[t][nt][2], run[t][nt][2]);
                            run[t][nt][3] = fmaf(-mb[t], am[t][nt][3], run[t][nt][3]);
                        }
                }
            } else if (RFMT == kFmtQ8 && u_fmt == RFMT) {
                // GGUF Q8_0: a group = 4 blocks of 32 rows (2 k-steps each, one
                // scale per column); codes become exact fp16 values, a block's
                // two k-steps are summed in fp32, then scaled
                const int nks = h.nb * 8;
                const int per = (nks + gwarps - 1) / gwarps;
                const int kb = gw * per, ke = min(kb + per, nks);
                float acc[2][NT][4];
                float sA[2] = {0.f, 0.f}, sB[2] = {0.f, 0.f};
                int blk = -1;  // current 32-row block (group * 4 + block)
                auto flush = [&]() {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            run[t][nt][0] = fmaf(sA[t], acc[t][nt][0], run[t][nt][0]);
                            run[t][nt][1] = fmaf(sA[t], acc[t][nt][1], run[t][nt][1]);
                            run[t][nt][2] = fmaf(sB[t], acc[t][nt][2], run[t][nt][2]);
                            run[t][nt][3] = fmaf(sB[t], acc[t][nt][3], run[t][nt][3]);
                        }
                };
                for (int kk = kb; kk < ke; ++kk) {
                    const int gr = kk >> 3, kl = kk & 7;
                    const uint8_t *gp = stage + (size_t)gr * kQ8GroupBytes;
                    if (gr * 4 + (kl >> 1) != blk) {
                        if (blk >= 0) flush();
                        blk = gr * 4 + (kl >> 1);
                        const __half *scp = reinterpret_cast<const __half *>(gp) + (kl >> 1) * 32;
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            sA[t] = __half2float(scp[t * 16 + g]);
                            sB[t] = __half2float(scp[t * 16 + g + 8]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int r = 0; r < 4; ++r) acc[t][nt][r] = 0.f;
                        }
                    }
                    const uint4 v = lds128(gp + kQ8ScaleBytes + kl * 512 + lane * 16);
                    const int ks = (h.b0 + gr) * 8 + kl;  // k-step within H
                    uint32_t bf0[NT], bf1[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const bool okx = xoff[nt] >= 0;
                        const __half *xr = xs + (okx ? xoff[nt] : 0) + 16 * ks;
                        bf0[nt] = okx ? lds32(xr) : 0u;
                        bf1[nt] = okx ? lds32(xr + 8) : 0u;
                    }
                    uint32_t a0[4], a1[4];
                    q8_frag(v.x, v.y, a0);
                    q8_frag(v.z, v.w, a1);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        if (nt < nact) {
                            mma_16816(acc[0][nt], a0, bf0[nt], bf1[nt]);
                            mma_16816(acc[1][nt], a1, bf0[nt], bf1[nt]);
                        }
                }
                if (blk >= 0) flush();
            } else {
                const int nb = h.nb;
                const int per = (nb + gwarps - 1) / gwarps;
                const int bb = gw * per, be = min(bb + per, nb);
                for (int b = bb; b < be; ++b) {
                    const int ks = h.b0 + b;
                    uint32_t bf0[NT], bf1[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const bool okx = xoff[nt] >= 0;
                        const __half *xr = xs + (okx ? xoff[nt] : 0) + 16 * ks;
                        bf0[nt] = okx ? lds32(xr) : 0u;
                        bf1[nt] = okx ? lds32(xr + 8) : 0u;
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint4 v = lds128(stage + ((size_t)b * 2 + t) * 512 + lane * 16);
                        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nact) mma_16816(run[t][nt], a, bf0[nt], bf1[nt]);
                    }
                }
            }
        } else if (n_e > 0 && h.kind == HK_DOWN) {
            const int nb = h.nb;
            const int per = (nb + gwarps - 1) / gwarps;
            const int bb = gw * per, be = min(bb + per, nb);
            for (int b = bb; b < be; ++b) {
                if (GG && u_fmt == RFMT) {
                    // GGUF Q8_0 down: block = one m-tile pair (one k-step of the
                    // unit's 16 rows), the lane's 8 codes of each tile; one scale
                    // per output for the unit's 32-row block
                    const uint4 v = lds128(stage + (size_t)b * 512 + lane * 16);
                    uint32_t a0[4], a1[4];
                    q8_frag(v.x, v.y, a0);
                    q8_frag(v.z, v.w, a1);
                    const int n0 = 32 * (h.b0 + b) + 4 * g;
                    const uint2 sv = *reinterpret_cast<const uint2 *>(sdcur + n0);
                    const float2 s01 = __half22float2(u32_as_h2(sv.x));
                    const float2 s23 = __half22float2(u32_as_h2(sv.y));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (nt < nact) {
                            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                            mma_16816(acc[0], a0, hb0[0][nt], hb1[0][nt]);
                            mma_16816(acc[1], a1, hb0[0][nt], hb1[0][nt]);
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int col = nt * 8 + 2 * q4 + hf;
                                if (col < n_e) {
                                    const float w = oscl[nt][hf];
                                    float4 o;
                                    o.x = acc[0][hf] * s01.x * w;
                                    o.y = acc[0][2 + hf] * s01.y * w;
                                    o.z = acc[1][hf] * s23.x * w;
                                    o.w = acc[1][2 + hf] * s23.y * w;
                                    atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)orow[nt][hf] * H + n0), o);
                                }
                            }
                        }
                    }
                } else if (W4R && u_fmt == FMT_W4) {
                    // block = 4/MS4 m-tiles (2/MS4 pairs), lane words [tile][ks]
                    constexpr int NPAIR = 2 / MS4;
                    const uint4 v = lds128(stage + (size_t)b * 512 + lane * 16);
                    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int pr = 0; pr < NPAIR; ++pr) {
                        uint32_t a[2][MS4][4];
#pragma unroll
                        for (int q = 0; q < 2; ++q)
#pragma unroll
                            for (int ks = 0; ks < MS4; ++ks) dequant_frag(words[(2 * pr + q) * MS4 + ks], a[q][ks]);
                        const int mt0 = (h.b0 + b) * (4 / MS4) + 2 * pr;
                        const int n0 = 32 * (mt0 >> 1) + 4 * g;
                        const uint2 sv = *reinterpret_cast<const uint2 *>(sdcur + n0);
                        const float2 s01 = __half22float2(u32_as_h2(sv.x));
                        const float2 s23 = __half22float2(u32_as_h2(sv.y));
                        float2 d01 = make_float2(0.f, 0.f), d23 = d01;  // ZP: 8 - zero point of outputs n0..n0+3
                        if (ZP) {
                            // the zero-point row keeps the column-block order of
                            // the pair's 32 outputs: output 32 Q + 4 m' + 2 q + h
                            // (m' < 8, tile q, row half h) sits at 16 q + 8 h + m'
                            const __half *zq = zdcur + (n0 - 4 * g);
                            d01 = make_float2(8.f - __half2float(zq[g]), 8.f - __half2float(zq[g + 8]));
                            d23 = make_float2(8.f - __half2float(zq[16 + g]), 8.f - __half2float(zq[24 + g]));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (nt < nact) {
                                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                                for (int q = 0; q < 2; ++q)
#pragma unroll
                                    for (int ks = 0; ks < MS4; ++ks)
                                        mma_16816(acc[q], a[q][ks], hb0[ks][nt], hb1[ks][nt]);
#pragma unroll
                                for (int hf = 0; hf < 2; ++hf) {
                                    const int col = nt * 8 + 2 * q4 + hf;
                                    if (col < n_e) {
                                        const float w = oscl[nt][hf];
                                        if (ZP) {
                                            const float hsm = hsum[nt][hf];
                                            acc[0][hf] = fmaf(d01.x, hsm, acc[0][hf]);
                                            acc[0][2 + hf] = fmaf(d01.y, hsm, acc[0][2 + hf]);
                                            acc[1][hf] = fmaf(d23.x, hsm, acc[1][hf]);
                                            acc[1][2 + hf] = fmaf(d23.y, hsm, acc[1][2 + hf]);
                                        }
                                        float4 o;
                                        o.x = acc[0][hf] * s01.x * w;
                                        o.y = acc[0][2 + hf] * s01.y * w;
                                        o.z = acc[1][hf] * s23.x * w;
                                        o.w = acc[1][2 + hf] * s23.y * w;
                                        atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)orow[nt][hf] * H + n0), o);
                                    }
                                }
                            }
                        }
                    }
                } else {
                    // block = one m-tile pair: [q][lane] x 16 B; a pair's second
                    // slice has its block nb blocks further on (k-step 1)
                    const bool two = (h.flags & HF_PAIR) != 0;
                    uint32_t a[2][2][4];
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            uint4 v = make_uint4(0u, 0u, 0u, 0u);
                            if (sl == 0 || two) v = lds128(stage + ((size_t)(sl * nb + b) * 2 + q) * 512 + lane * 16);
                            a[sl][q][0] = v.x;
                            a[sl][q][1] = v.y;
                            a[sl][q][2] = v.z;
                            a[sl][q][3] = v.w;
                        }
                    const int n0 = 32 * (h.b0 + b) + 4 * g;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (nt < nact) {
                            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                mma_16816(acc[q], a[0][q], hb0[0][nt], hb1[0][nt]);
                                if (two) mma_16816(acc[q], a[1][q], hb0[1][nt], hb1[1][nt]);
                            }
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int col = nt * 8 + 2 * q4 + hf;
                                if (col < n_e) {
                                    const float w = oscl[nt][hf];
                                    float4 o;
                                    o.x = acc[0][hf] * w;
                                    o.y = acc[0][2 + hf] * w;
                                    o.z = acc[1][hf] * w;
                                    o.w = acc[1][2 + hf] * w;
                                    atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)orow[nt][hf] * H + n0), o);
                                }
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (h.flags & HF_GU_LAST) {
            // cross-warp reduction of the (sub-)unit's gate/up partial sums
            // (shared-memory atomics into the group's buffer: gate rows [0, S),
            // up rows [S, 2S); an FP16 pair's second slice at row offset 16)
            const int S = u_S;
            const bool f16u = u_fmt == FMT_F16;
            const int roff = (h.flags & HF_SUB1) ? 16 : 0;
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                if (f16u ? t < 2 : t * 16 < 2 * S) {
                    const int ra = (f16u ? t * S + roff : t * 16) + g, rb = ra + 8;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int col = nt * 8 + 2 * q4;
                        if (col < n_e) {
                            atomicAdd(red + ra * rs + col, run[t][nt][0]);
                            atomicAdd(red + rb * rs + col, run[t][nt][2]);
                            if (col + 1 < n_e) {
                                atomicAdd(red + ra * rs + col + 1, run[t][nt][1]);
                                atomicAdd(red + rb * rs + col + 1, run[t][nt][3]);
                            }
                        }
#pragma unroll
                        for (int r = 0; r < 4; ++r) run[t][nt][r] = 0.f;
                    }
                }
            }
        }
        if (h.flags & HF_GU_FINAL) {
            // SiLU, h -> fp16 fragments; the buffer is left zeroed for the
            // group's next unit
            const int S = u_S;
            if (W4R || GG) cp_async_wait_all();  // this thread's share of the down-scale (and zero-point) row
            group_sync(p, gs, abort_flag);
            // only the unit's n_e token columns hold sums (the others stay
            // zero); h columns past n_e feed output columns that are never
            // stored, so they are left as they are
            for (int idx = gtid; idx < S * n_e; idx += gwarps * 32) {
                const int i = idx / n_e, col = idx - i * n_e;
                const float gv = red[(size_t)i * rs + col], uv = red[(size_t)(S + i) * rs + col];
                red[(size_t)i * rs + col] = 0.f;
                red[(size_t)(S + i) * rs + col] = 0.f;
                hs[col * kHsStride + i] = __float2half_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
            }
            group_sync(p, gs, abort_flag);
            const int kst = S / 16;
#pragma unroll
            for (int ks = 0; ks < KH; ++ks)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int col = nt * 8 + g;
                    const bool okh = ks < kst && col < npad;
                    const __half *hr = hs + (okh ? col * kHsStride + 16 * ks + 2 * q4 : 0);
                    hb0[ks][nt] = okh ? lds32(hr) : 0u;
                    hb1[ks][nt] = okh ? lds32(hr + 8) : 0u;
                }
            if (ZP) {  // this lane's output columns' sums of h over the unit's rows
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int col = nt * 8 + 2 * q4 + hf;
                        float sum = 0.f;
                        if (col < n_e) {
                            const __half2 *hr2 = reinterpret_cast<const __half2 *>(hs + col * kHsStride);
                            for (int i = 0; i < S / 2; ++i) {
                                const float2 f = __half22float2(hr2[i]);
                                sum += f.x + f.y;
                            }
                        }
                        hsum[nt][hf] = sum;
                    }
            }
        }
        ++it;
    }

    // Completion: the last kEpiBlocks blocks to finish wait until every block
    // has (their own work is done; all blocks of the grid are resident) and
    // each turns its share of the fp32 sums into the fp16 output and clears
    // it; the last of them to leave resets the counters.
    group_sync(p, as, abort_flag);
    if (ctid == 0) {
        __threadfence();
        misc[1] = (int)atomicAdd(&p.hdr->done_ticket, 1u);
    }
    group_sync(p, as, abort_flag);
    const int nhelp = (int)gridDim.x < kEpiBlocks ? (int)gridDim.x : kEpiBlocks;
    const int part = misc[1] - ((int)gridDim.x - nhelp);
    if (part >= 0) {
        if (ctid == 0) {
            // bounded wait for the remaining blocks
            const volatile uint32_t *dt = &p.hdr->done_ticket;
            const uint64_t t0 = global_timer_ns();
            bool ok = true;
            while (*dt < gridDim.x) {
                if (*abort_flag || global_timer_ns() - t0 > p.wait_budget_ns) {
                    record_timeout(&p.hdr->status, SITE_ENGINE);
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
            misc[2] = ok;
            __threadfence();
        }
        group_sync(p, as, abort_flag);
        if (p.mode == MODE_LAYER && misc[2]) {
            // rows of this part, read in batches of 16 float4 per thread with
            // all loads of a batch in flight before any store
            const int n4 = p.T * H / 4;
            const int per = (n4 + nhelp - 1) / nhelp;
            const int lo = part * per, hi = min(n4, lo + per);
            constexpr int kNth = kConsumerWarps * 32, kBatch = 16;
            float4 *acc4 = reinterpret_cast<float4 *>(p.yout);
            for (int i0 = lo + ctid; i0 < hi; i0 += kNth * kBatch) {
                float4 v[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = i0 + j * kNth;
                    v[j] = idx < hi ? __ldcg(acc4 + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = i0 + j * kNth;
                    if (idx < hi) {
                        uint2 o;
                        o.x = h2_as_u32(__floats2half2_rn(v[j].x, v[j].y));
                        o.y = h2_as_u32(__floats2half2_rn(v[j].z, v[j].w));
                        reinterpret_cast<uint2 *>(p.out)[idx] = o;
                        __stcg(acc4 + idx, make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                }
            }
        }
        group_sync(p, as, abort_flag);
        if (ctid == 0) {
            __threadfence();
            if (atomicAdd(&p.hdr->exit_ticket, 1u) == (uint32_t)nhelp - 1) {
                // no fence after these: the launch that follows reads them only
                // after this one has completed
                p.hdr->work_counter = 0;
                p.hdr->done_ticket = 0;
                p.hdr->exit_ticket = 0;
            }
        }
    }
}

// token tables for the unit calls: row = sorted position, scale = 1
__global__ void __launch_bounds__(64) tables_kernel(const int32_t *offsets, const int32_t *sorted_slots,
                                                    const int32_t *active, const int32_t *n_active, int T, int k,
                                                    int E, TokTable *tables) {
    int na = *n_active;
    na = na < 0 ? 0 : (na > E ? E : na);
    for (int a = blockIdx.x; a < na; a += gridDim.x) {
        const int e = active[a];
        if (e < 0 || e >= E) continue;
        const int o0 = offsets[e];
        int n = offsets[e + 1] - o0;
        n = (n < 0 || n > T) ? 0 : n;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int pidx = o0 + i;
            int s = (pidx >= 0 && pidx < T * k) ? sorted_slots[pidx] : 0;
            s = (s >= 0 && s < T * k) ? s : 0;
            TokEntry te;
            te.tok = s / k;
            te.row = pidx;
            te.scale = 1.0f;
            te.pad = 0;
            tables[e].e[i] = te;
        }
        if (threadIdx.x == 0) tables[e].n = n;
    }
}

int launch_tables(const int32_t *offsets, const int32_t *sorted_slots, const int32_t *active, const int32_t *n_active,
                  int T, int k, int E, TokTable *tables, cudaStream_t s) {
    tables_kernel<<<E < 64 ? E : 64, 64, 0, s>>>(offsets, sorted_slots, active, n_active, T, k, E, tables);
    return record_launch(cudaGetLastError());
}

// ------------------------------------------------------------ launching --
// Token tiles of 8 an expert launch instance carries: 1, 2, 3, 5 (FP16 only;
// the other formats take 5 as 8) or 8.  Narrower instances need fewer
// registers: the 2-tile ones (9-16 tokens) do not spill (FP16: 108 registers
// instead of 132): verify at 9 tokens 3% faster, INT4 draft batches of 16
// tokens 27%; the 5-tile FP16 one (25-40 tokens, 162 registers, no spill)
// took verify at 33 tokens from 372 to 257 us against the spilling 8-tile one.
int engine_nt(int T) { return T <= 8 ? 1 : (T <= 16 ? 2 : (T <= 24 ? 3 : (T <= 40 ? 5 : 8))); }

// Geometry: two consumer groups of two stages each (two units in parallel,
// each double-buffered), with the largest chunk (a multiple of 1 KB, at most
// 4 kChunk) that shared memory holds: the bytes a block keeps in flight bound
// the launch, and bigger chunks mean fewer producer steps.  Where that chunk
// would be small (wide activation rows: below kGroupSplitMin), one group of
// two stages of twice the size is faster (Phi-3.5-MoE-shaped verify: 455 ->
// 434 us on GB300; DeepSeek-V2-Lite-shaped, 36 KB chunks: two groups).  Below
// kChunk per chunk even then, one group with as many kChunk stages as fit.
constexpr int kGroupSplitMin = 28 * 1024;
static int fit_chunk(int T, int H, int npad, int smax, bool w4, int G, int nsg, bool zp, int kqs) {
    const int base = smem_layout(T, H, npad, smax, w4, G, nsg, 0, zp, kqs).total;
    int chunk = ((kSmemLimit - base) / (G * nsg) - meta_bytes_for(T)) / 1024 * 1024;
    return chunk > 4 * kChunk ? 4 * kChunk : chunk;
}
static bool choose_geometry(int T, int H, int npad, int smax, bool w4, int &G, int &nsg, int &bytes, int &chunk,
                            bool zp = false, int kqs = 0) {
    G = 2;
    nsg = 2;
    chunk = fit_chunk(T, H, npad, smax, w4, G, nsg, zp, kqs);
    if (chunk < kGroupSplitMin) {
        const int c1 = fit_chunk(T, H, npad, smax, w4, 1, 2, zp, kqs);
        if (c1 >= kChunk && c1 > chunk) {
            G = 1;
            chunk = c1;
        }
    }
    if (chunk >= kChunk) {
        bytes = smem_layout(T, H, npad, smax, w4, G, nsg, chunk, zp, kqs).total;
        return bytes <= kSmemLimit;
    }
    G = 1;
    chunk = kChunk;
    for (nsg = 12; nsg >= 2; --nsg) {
        const SmemLayout L = smem_layout(T, H, npad, smax, w4, G, nsg, chunk, zp, kqs);
        if (L.total <= kSmemLimit) {
            bytes = L.total;
            return true;
        }
    }
    return false;
}

// Loads the kernel instance on the current device and raises its dynamic
// shared-memory limit, once per device.
template <int RFMT, int MS4, int NT>
static int configure_engine() {
    static int configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPX_ERR_CUDA;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(engine_kernel<RFMT, MS4, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return record_launch(e);
        configured[dev] = 1;
    }
    return SPX_OK;
}

template <int RFMT, int MS4, int NT>
static int launch_engine_t(const EngineParams &p0, cudaStream_t s, bool pdl) {
    EngineParams p = p0;
    const int sms = device_sm_count();
    if (sms <= 0) return SPX_ERR_CUDA;
    const bool w4 = (RFMT == FMT_W4 || RFMT == FMT_W4Z || RFMT == kFmtQ8 || RFMT == kFmtQ2K || RFMT == kFmtQ4K) &&
                    p.routed_enabled;
    const int smax = engine_smax(w4, p.S);
    const int kqs = RFMT == kFmtQ2K ? 16 : RFMT == kFmtQ4K ? 32 : 0;
    int G, nsg, bytes, chunk;
    if (!choose_geometry(p.T, p.H, p.npad, smax, w4, G, nsg, bytes, chunk, RFMT == FMT_W4Z, kqs))
        return SPX_ERR_UNSUPPORTED;
    p.groups = G;
    p.nstages = nsg;
    p.chunk = chunk;
    const int st = configure_engine<RFMT, MS4, NT>();
    if (st) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return record_launch(cudaLaunchKernelEx(&cfg, engine_kernel<RFMT, MS4, NT>, p));
}

int launch_engine(const EngineParams &p, cudaStream_t s, bool pdl) {
    const int nt = engine_nt(p.T);
    if (p.routed_enabled && p.routed_fmt == kFmtQ8) {
        if (nt == 1) return launch_engine_t<kFmtQ8, 1, 1>(p, s, pdl);
        if (nt == 2) return launch_engine_t<kFmtQ8, 1, 2>(p, s, pdl);
        if (nt == 3) return launch_engine_t<kFmtQ8, 1, 3>(p, s, pdl);
        return launch_engine_t<kFmtQ8, 1, 8>(p, s, pdl);
    }
    if (p.routed_enabled && p.routed_fmt == kFmtQ2K) {
        if (nt == 1) return launch_engine_t<kFmtQ2K, 1, 1>(p, s, pdl);
        if (nt == 2) return launch_engine_t<kFmtQ2K, 1, 2>(p, s, pdl);
        if (nt == 3) return launch_engine_t<kFmtQ2K, 1, 3>(p, s, pdl);
        return launch_engine_t<kFmtQ2K, 1, 8>(p, s, pdl);
    }
    if (p.routed_enabled && p.routed_fmt == kFmtQ4K) {
        if (nt == 1) return launch_engine_t<kFmtQ4K, 1, 1>(p, s, pdl);
        if (nt == 2) return launch_engine_t<kFmtQ4K, 1, 2>(p, s, pdl);
        if (nt == 3) return launch_engine_t<kFmtQ4K, 1, 3>(p, s, pdl);
        return launch_engine_t<kFmtQ4K, 1, 8>(p, s, pdl);
    }
    if (p.routed_enabled && p.routed_fmt == FMT_W4 && p.w4_zeros) {
        if (p.S == 32) {
            if (nt == 1) return launch_engine_t<FMT_W4Z, 2, 1>(p, s, pdl);
            if (nt == 2) return launch_engine_t<FMT_W4Z, 2, 2>(p, s, pdl);
            if (nt == 3) return launch_engine_t<FMT_W4Z, 2, 3>(p, s, pdl);
            return SPX_ERR_UNSUPPORTED;
        }
        if (nt == 1) return launch_engine_t<FMT_W4Z, 1, 1>(p, s, pdl);
        if (nt == 2) return launch_engine_t<FMT_W4Z, 1, 2>(p, s, pdl);
        if (nt == 3) return launch_engine_t<FMT_W4Z, 1, 3>(p, s, pdl);
        return launch_engine_t<FMT_W4Z, 1, 8>(p, s, pdl);
    }
    if (p.routed_enabled && p.routed_fmt == FMT_W4) {
        if (p.S == 32) {
            if (nt == 1) return launch_engine_t<FMT_W4, 2, 1>(p, s, pdl);
            if (nt == 2) return launch_engine_t<FMT_W4, 2, 2>(p, s, pdl);
            if (nt == 3) return launch_engine_t<FMT_W4, 2, 3>(p, s, pdl);
            return SPX_ERR_UNSUPPORTED;  // INT4 slices of 32 columns take at most 24 tokens per expert
        }
        if (nt == 1) return launch_engine_t<FMT_W4, 1, 1>(p, s, pdl);
        if (nt == 2) return launch_engine_t<FMT_W4, 1, 2>(p, s, pdl);
        if (nt == 3) return launch_engine_t<FMT_W4, 1, 3>(p, s, pdl);
        return launch_engine_t<FMT_W4, 1, 8>(p, s, pdl);
    }
    if (nt == 1) return launch_engine_t<FMT_F16, 1, 1>(p, s, pdl);
    if (nt == 2) return launch_engine_t<FMT_F16, 1, 2>(p, s, pdl);
    if (nt == 3) return launch_engine_t<FMT_F16, 1, 3>(p, s, pdl);
    if (nt == 5) return launch_engine_t<FMT_F16, 1, 5>(p, s, pdl);
    return launch_engine_t<FMT_F16, 1, 8>(p, s, pdl);
}

int engine_preload() {
    int st = SPX_OK;
    if (!st) st = configure_engine<FMT_W4, 2, 1>();
    if (!st) st = configure_engine<FMT_W4, 2, 2>();
    if (!st) st = configure_engine<FMT_W4, 1, 2>();
    if (!st) st = configure_engine<FMT_W4Z, 2, 2>();
    if (!st) st = configure_engine<FMT_W4Z, 1, 2>();
    if (!st) st = configure_engine<kFmtQ8, 1, 2>();
    if (!st) st = configure_engine<kFmtQ2K, 1, 2>();
    if (!st) st = configure_engine<kFmtQ4K, 1, 2>();
    if (!st) st = configure_engine<FMT_W4, 2, 3>();
    if (!st) st = configure_engine<FMT_W4, 1, 1>();
    if (!st) st = configure_engine<FMT_W4, 1, 3>();
    if (!st) st = configure_engine<FMT_W4, 1, 8>();
    if (!st) st = configure_engine<FMT_W4Z, 2, 1>();
    if (!st) st = configure_engine<FMT_W4Z, 2, 3>();
    if (!st) st = configure_engine<FMT_W4Z, 1, 1>();
    if (!st) st = configure_engine<FMT_W4Z, 1, 3>();
    if (!st) st = configure_engine<FMT_W4Z, 1, 8>();
    if (!st) st = configure_engine<kFmtQ8, 1, 1>();
    if (!st) st = configure_engine<kFmtQ8, 1, 3>();
    if (!st) st = configure_engine<kFmtQ8, 1, 8>();
    if (!st) st = configure_engine<kFmtQ2K, 1, 1>();
    if (!st) st = configure_engine<kFmtQ2K, 1, 3>();
    if (!st) st = configure_engine<kFmtQ2K, 1, 8>();
    if (!st) st = configure_engine<kFmtQ4K, 1, 1>();
    if (!st) st = configure_engine<kFmtQ4K, 1, 3>();
    if (!st) st = configure_engine<kFmtQ4K, 1, 8>();
    if (!st) st = configure_engine<FMT_F16, 1, 1>();
    if (!st) st = configure_engine<FMT_F16, 1, 2>();
    if (!st) st = configure_engine<FMT_F16, 1, 5>();
    if (!st) st = configure_engine<FMT_F16, 1, 3>();
    if (!st) st = configure_engine<FMT_F16, 1, 8>();
    cudaFuncAttributes fa;
    if (!st) st = record_launch(cudaFuncGetAttributes(&fa, tables_kernel));
    return st;
}

int engine_fits(int T, int H, int fmt, int S) {
    const int npad = 8 * ((T + 7) / 8);
    const bool zp = fmt == FMT_W4Z;
    const bool w4 = fmt == FMT_W4 || zp || fmt == kFmtQ8 || fmt == kFmtQ2K || fmt == kFmtQ4K;  // down-scale rows
    const int kqs = fmt == kFmtQ2K ? 16 : fmt == kFmtQ4K ? 32 : 0;
    if (kqs && H % 256) return 0;
    if (w4 && S == 32 && engine_nt(T) > 3) return 0;  // 32-column slices: at most 3 token tiles
    int G, nsg, bytes, chunk;
    return choose_geometry(T, H, npad, engine_smax(w4, S), w4, G, nsg, bytes, chunk, zp, kqs) ? 1 : 0;
}

}  // namespace spx
