// spx_engine.cu -- the expert MLP launch shared by the INT4 draft path, the
// FP16 verify path, the shared expert and the composite layer.
//
// Method (ai.info summary of the Specter paper, Key Contributions 4 and
// "Methodology in Plain English"; richland.au post, "What shipped"):
//  - draft: all active experts' INT4 (GPTQ, group 128) MLPs in ONE launch,
//    dequantised in-register and multiplied with fp16 activations (W4A16);
//  - verify: tokens routed to the same expert are packed together so that each
//    expert's FP16 weights are read once and multiplied by all of its tokens
//    as one dense tensor-core product (the "expert-wise reordering");
//  - the FP16 shared expert runs in the same launch; it does not depend on
//    routing, so it is queued first.
//
// GB300 design.  Persistent grid, one block per SM (152 on GB300), each block
// = 8 consumer warps + 1 producer warp.  Work is a dynamic queue of "units":
// one unit = one expert's slice of S intermediate columns, so the gate/up
// reduction over H and the SiLU stay inside one block and the down
// projection's partial sums over the slices are added into fp32 outputs with
// vector atomics (no grid-wide barrier, no spin on other blocks).  A unit is
// contiguous in HBM (repacked once at load time) and streamed by the producer
// with 16 KB bulk copies (TMA engine) into a ring of shared-memory stages
// guarded by mbarriers; consumers read their mma.sync A fragments with
// conflict-free 16-byte shared loads, dequantise INT4 in registers, and use
// the activations (also in shared memory) as the B operand.
#include "spx_internal.cuh"

#include <math.h>

namespace spx {

enum : int { HK_SCALES = 0, HK_GU = 1, HK_DOWN = 2, HK_DONE = 3 };
enum : int { HF_UNIT_START = 1, HF_GU_LAST = 2 };
enum : int { MODE_SORTED = 0, MODE_ACC = 1, MODE_LAYER = 2 };
enum : int { FMT_W4 = 0, FMT_F16 = 1 };

struct __align__(16) ChunkHeader {
    int unit;
    int kind;
    int b0;
    int nb_flags;  // blocks | flags << 16
};


struct SmemLayout {
    int bars, hdrs, tok, misc, sc, red, hs, xs, ring, total;
    int xs_stride;  // halves per activation row
};

constexpr int kHsStride = 40;  // halves per intermediate row (32 + 8 pad)

__host__ __device__ inline SmemLayout smem_layout(int T, int H, int npad, int nstages) {
    SmemLayout L;
    int o = 0;
    L.bars = o;
    o += (2 * nstages + 1) * 8;
    o = (o + 15) & ~15;
    L.hdrs = o;
    o += nstages * 16;
    L.tok = o;
    o += 4 * kMaxT * 4;  // tok_x, tok_row, tok_scale, gamma
    L.misc = o;
    o += 64;
    L.sc = o;
    o += (H / 128) * 64 * 2;  // up to 2*32 columns of fp16 scales per group
    o = (o + 15) & ~15;
    L.red = o;
    o += 64 * npad * 4;
    L.hs = o;
    o += npad * kHsStride * 2;
    o = (o + 15) & ~15;
    L.xs = o;
    L.xs_stride = H + 8;
    o += T * (H + 8) * 2;
    o = (o + 127) & ~127;
    L.ring = o;
    o += nstages * kChunk;
    L.total = o;
    return L;
}

struct UnitInfo {
    int fmt, S, e, i0, n_e, is_shared;
    const uint8_t *base;
};

__device__ __forceinline__ bool decode_unit(const EngineParams &p, int u, int n_sh, UnitInfo &ui) {
    if (u < n_sh) {
        ui.fmt = FMT_F16;
        ui.S = kF16S;
        ui.e = 0;
        ui.i0 = u * kF16S;
        ui.is_shared = 1;
        ui.n_e = p.T;
        ui.base = p.shared + (size_t)u * f16_unit_bytes(p.H);
        return true;
    }
    const int spe = p.I / p.S;
    const int r = u - n_sh;
    const int a = r / spe, j = r - a * spe;
    if (a >= p.E) return false;
    const int e = __ldcg(p.active + a);
    if (e < 0 || e >= p.E) return false;
    ui.fmt = p.routed_fmt;
    ui.S = p.S;
    ui.e = e;
    ui.i0 = j * p.S;
    ui.is_shared = 0;
    const int o0 = __ldcg(p.offsets + e), o1 = __ldcg(p.offsets + e + 1);
    ui.n_e = (o0 >= 0 && o1 >= o0 && o1 - o0 <= p.T && o1 <= p.T * p.k) ? o1 - o0 : 0;
    const size_t ub = p.routed_fmt == FMT_W4 ? w4_unit_bytes(p.H, p.S) : f16_unit_bytes(p.H);
    ui.base = p.routed + ((size_t)e * spe + j) * ub;
    return true;
}

// ------------------------------------------------------------- producer --
__device__ void producer_loop(const EngineParams &p, uint8_t *smem, const SmemLayout &L) {
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + p.nstages;
    ChunkHeader *hdrs = reinterpret_cast<ChunkHeader *>(smem + L.hdrs);
    uint8_t *ring = smem + L.ring;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc);
    const uint64_t pol = policy_evict_first();
    const int n_sh = p.shared ? p.I_s / kF16S : 0;
    int n_total = -1;
    uint32_t it = 0;

    auto emit = [&](int unit, int kind, int b0, int nb, int flags, const uint8_t *src, uint32_t bytes) -> bool {
        const int st = it % p.nstages;
        const uint32_t round = it / p.nstages;
        if (!mbar_wait_bounded(&empty[st], (round & 1) ^ 1, abort_flag, &p.hdr->status, p.wait_budget_ns))
            return false;
        ChunkHeader h;
        h.unit = unit;
        h.kind = kind;
        h.b0 = b0;
        h.nb_flags = nb | (flags << 16);
        hdrs[st] = h;
        if (bytes) {
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s(ring + (size_t)st * kChunk, src, bytes, &full[st], pol);
        } else {
            mbar_arrive(&full[st]);
        }
        ++it;
        return true;
    };

    bool ok = true;
    while (ok) {
        const int u = (int)atomicAdd(&p.hdr->work_counter, 1u);
        if (u >= n_sh) {
            if (n_total < 0) {
                int nr = 0;
                if (p.routed_enabled) {
                    griddep_wait();
                    int na = __ldcg(p.n_active);
                    na = na < 0 ? 0 : (na > p.E ? p.E : na);
                    nr = na * (p.I / p.S);
                }
                n_total = n_sh + nr;
            }
            if (u >= n_total) break;
        }
        UnitInfo ui;
        if (!decode_unit(p, u, n_sh, ui)) continue;
        const int H = p.H;
        if (ui.fmt == FMT_W4) {
            const int S = ui.S;
            const uint32_t scb = (uint32_t)w4_sc_bytes(H, S);
            ok = emit(u, HK_SCALES, 0, 0, HF_UNIT_START, ui.base, scb);
            const uint8_t *gu = ui.base + scb;
            const int nbg = (int)(w4_gu_bytes(H, S) / 512);
            for (int b = 0; ok && b < nbg; b += kChunk / 512) {
                const int nb = min(kChunk / 512, nbg - b);
                ok = emit(u, HK_GU, b, nb, b + nb == nbg ? HF_GU_LAST : 0, gu + (size_t)b * 512, nb * 512);
            }
            const uint8_t *dn = gu + w4_gu_bytes(H, S);
            const int nbd = (int)(w4_dn_bytes(H, S) / 512);
            for (int b = 0; ok && b < nbd; b += kChunk / 512) {
                const int nb = min(kChunk / 512, nbd - b);
                ok = emit(u, HK_DOWN, b, nb, 0, dn + (size_t)b * 512, nb * 512);
            }
        } else {
            const int nbg = H / 16;  // one k-step (1 KB) per block
            for (int b = 0; ok && b < nbg; b += kChunk / 1024) {
                const int nb = min(kChunk / 1024, nbg - b);
                const int fl = (b == 0 ? HF_UNIT_START : 0) | (b + nb == nbg ? HF_GU_LAST : 0);
                ok = emit(u, HK_GU, b, nb, fl, ui.base + (size_t)b * 1024, nb * 1024);
            }
            const uint8_t *dn = ui.base + f16_gu_bytes(H);
            const int nbd = H / 32;  // one m-tile pair (1 KB) per block
            for (int b = 0; ok && b < nbd; b += kChunk / 1024) {
                const int nb = min(kChunk / 1024, nbd - b);
                ok = emit(u, HK_DOWN, b, nb, 0, dn + (size_t)b * 1024, nb * 1024);
            }
        }
    }
    if (ok) emit(-1, HK_DONE, 0, 0, 0, nullptr, 0);
    // Drain: every issued copy has been waited on by the consumers unless the
    // block aborted; in that case wait (bounded) for the copies in flight.
    if (*abort_flag) {
        const uint32_t first = it > (uint32_t)p.nstages ? it - p.nstages : 0;
        for (uint32_t j = first; j < it; ++j) {
            const int st = j % p.nstages;
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[st], (j / p.nstages) & 1) && global_timer_ns() - t0 < 100000000ull) {
            }
        }
    }
}

// ------------------------------------------------------------ consumers --
struct ConsumerCtx {
    uint64_t *full, *empty, *csync;
    ChunkHeader *hdrs;
    uint8_t *ring;
    int *tok_x, *tok_row;
    float *tok_scale, *gamma;
    volatile int *abort_flag;
    int *misc;
    __half *sc, *hs, *xs;
    float *red;
    int xs_stride;
    uint32_t csync_phase;
};

__device__ __forceinline__ void cons_sync(const EngineParams &p, ConsumerCtx &c) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(c.csync);
    mbar_wait_bounded(c.csync, c.csync_phase & 1, c.abort_flag, &p.hdr->status, p.wait_budget_ns);
    c.csync_phase ^= 1;
    __syncwarp();
}

// gate/up part of one chunk: this warp's blocks; partial sums folded into red
template <int MS4, int NT>
__device__ __forceinline__ void process_gu(const EngineParams &p, ConsumerCtx &c, const UnitInfo &ui,
                                           const uint8_t *stage, int b0, int nb) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q4 = lane & 3;
    const int per = (nb + kConsumerWarps - 1) / kConsumerWarps;
    const int bb = warp * per, be = min(bb + per, nb);
    if (bb >= be) return;
    const int npad = p.npad;
    const int ntb = (ui.n_e + 8 * NT - 1) / (8 * NT);
    for (int tb = 0; tb < ntb; ++tb) {
        const int col0 = tb * 8 * NT;
        const int nact = min(NT, (ui.n_e - col0 + 7) / 8);
        const __half *xr[NT];
        bool have[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = col0 + nt * 8 + g;
            have[nt] = col < ui.n_e;
            xr[nt] = c.xs + (size_t)(have[nt] ? c.tok_x[col] : 0) * c.xs_stride + 2 * q4;
        }
        if (ui.fmt == FMT_W4) {
            constexpr int KB = 2 / MS4, NTILE = 2 * MS4;
            const int S = ui.S;  // == 16 * MS4
            float acc[NTILE][NT][4];
            int grp = -1;
            auto fold = [&]() {
#pragma unroll
                for (int t = 0; t < NTILE; ++t) {
                    const int ra = t * 16 + g, rb = ra + 8;
                    const float sa = __half2float(c.sc[grp * 2 * S + ra]);
                    const float sb = __half2float(c.sc[grp * 2 * S + rb]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (nt < nact) {
                            const int col = col0 + nt * 8 + 2 * q4;
                            atomicAdd(&c.red[ra * npad + col], sa * acc[t][nt][0]);
                            atomicAdd(&c.red[ra * npad + col + 1], sa * acc[t][nt][1]);
                            atomicAdd(&c.red[rb * npad + col], sb * acc[t][nt][2]);
                            atomicAdd(&c.red[rb * npad + col + 1], sb * acc[t][nt][3]);
                        }
                    }
                }
            };
            for (int b = bb; b < be; ++b) {
                const uint4 v = lds128(stage + (size_t)b * 512 + lane * 16);
                const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int ki = 0; ki < KB; ++ki) {
                    const int ks = (b0 + b) * KB + ki;
                    const int gnew = ks >> 3;
                    if (gnew != grp) {
                        if (grp >= 0) fold();
#pragma unroll
                        for (int t = 0; t < NTILE; ++t)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int r = 0; r < 4; ++r) acc[t][nt][r] = 0.f;
                        grp = gnew;
                    }
                    uint32_t bf0[NT], bf1[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        bf0[nt] = have[nt] ? lds32(xr[nt] + 16 * ks) : 0u;
                        bf1[nt] = have[nt] ? lds32(xr[nt] + 16 * ks + 8) : 0u;
                    }
#pragma unroll
                    for (int t = 0; t < NTILE; ++t) {
                        uint32_t a[4];
                        dequant_frag(words[ki * NTILE + t], a);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nact) mma_16816(acc[t][nt], a, bf0[nt], bf1[nt]);
                    }
                }
            }
            if (grp >= 0) fold();
        } else {
            float acc[2][NT][4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[t][nt][r] = 0.f;
            for (int b = bb; b < be; ++b) {
                const int ks = b0 + b;
                uint32_t bf0[NT], bf1[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    bf0[nt] = have[nt] ? lds32(xr[nt] + 16 * ks) : 0u;
                    bf1[nt] = have[nt] ? lds32(xr[nt] + 16 * ks + 8) : 0u;
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint4 v = lds128(stage + ((size_t)b * 2 + t) * 512 + lane * 16);
                    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        if (nt < nact) mma_16816(acc[t][nt], a, bf0[nt], bf1[nt]);
                }
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int ra = t * 16 + g, rb = ra + 8;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (nt < nact) {
                        const int col = col0 + nt * 8 + 2 * q4;
                        atomicAdd(&c.red[ra * npad + col], acc[t][nt][0]);
                        atomicAdd(&c.red[ra * npad + col + 1], acc[t][nt][1]);
                        atomicAdd(&c.red[rb * npad + col], acc[t][nt][2]);
                        atomicAdd(&c.red[rb * npad + col + 1], acc[t][nt][3]);
                    }
                }
            }
        }
    }
}

// h = silu(g) * u for the unit's S columns and all token columns; rounds to
// fp16 (the down product's B operand) and re-zeroes the scratch.
__device__ __forceinline__ void compute_h(const EngineParams &p, ConsumerCtx &c, const UnitInfo &ui) {
    const int S = ui.S, npad = p.npad;
    for (int idx = threadIdx.x; idx < S * npad; idx += kConsumerWarps * 32) {
        const int i = idx / npad, col = idx - i * npad;
        const float gv = c.red[i * npad + col];
        const float uv = c.red[(S + i) * npad + col];
        const float h = gv / (1.0f + __expf(-gv)) * uv;
        c.hs[col * kHsStride + i] = __float2half_rn(h);
        c.red[i * npad + col] = 0.f;
        c.red[(S + i) * npad + col] = 0.f;
    }
}

// down part of one chunk: y[token][n] += scale_token * sum_i W_d[i][n] h[i]
template <int MS4, int NT>
__device__ __forceinline__ void process_down(const EngineParams &p, ConsumerCtx &c, const UnitInfo &ui,
                                             const uint8_t *stage, int b0, int nb) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q4 = lane & 3;
    const int per = (nb + kConsumerWarps - 1) / kConsumerWarps;
    const int bb = warp * per, be = min(bb + per, nb);
    if (bb >= be) return;
    const int H = p.H;
    const int ntb = (ui.n_e + 8 * NT - 1) / (8 * NT);
    const __half *sdrow = nullptr;
    if (ui.fmt == FMT_W4) sdrow = p.w4_sdown + ((size_t)ui.e * (p.I / 128) + ui.i0 / 128) * H;
    constexpr int MSMAX = MS4 > 1 ? MS4 : 1;
    for (int tb = 0; tb < ntb; ++tb) {
        const int col0 = tb * 8 * NT;
        const int nact = min(NT, (ui.n_e - col0 + 7) / 8);
        uint32_t hb0[MSMAX][NT], hb1[MSMAX][NT];
        const int kst = ui.S / 16;
#pragma unroll
        for (int ks = 0; ks < MSMAX; ++ks)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = col0 + nt * 8 + g;
                const bool ok = ks < kst && col < p.npad;
                const __half *hr = c.hs + col * kHsStride + 16 * ks + 2 * q4;
                hb0[ks][nt] = ok ? lds32(hr) : 0u;
                hb1[ks][nt] = ok ? lds32(hr + 8) : 0u;
            }
        for (int b = bb; b < be; ++b) {
            // tile pairs in this block: INT4 MS4=2 -> 1 pair, MS4=1 -> 2 pairs; FP16 -> 1 pair
            uint32_t words[4];
            int npairs;
            if (ui.fmt == FMT_W4) {
                const uint4 v = lds128(stage + (size_t)b * 512 + lane * 16);
                words[0] = v.x;
                words[1] = v.y;
                words[2] = v.z;
                words[3] = v.w;
                npairs = 2 / kst;
            } else {
                npairs = 1;
            }
            for (int pr = 0; pr < npairs; ++pr) {
                int mt0;
                float acc[2][NT][4];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[q][nt][r] = 0.f;
                float sd[4] = {1.f, 1.f, 1.f, 1.f};
                if (ui.fmt == FMT_W4) {
                    const int MB = 4 / kst;
                    mt0 = (b0 + b) * MB + 2 * pr;
                    const int n0 = 32 * (mt0 >> 1) + 4 * g;
                    const uint2 sv = __ldg(reinterpret_cast<const uint2 *>(sdrow + n0));
                    const float2 s01 = __half22float2(u32_as_h2(sv.x));
                    const float2 s23 = __half22float2(u32_as_h2(sv.y));
                    sd[0] = s01.x;
                    sd[1] = s01.y;
                    sd[2] = s23.x;
                    sd[3] = s23.y;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int ks = 0; ks < MSMAX; ++ks) {
                            if (ks < kst) {
                                uint32_t a[4];
                                dequant_frag(words[(2 * pr + q) * kst + ks], a);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    if (nt < nact) mma_16816(acc[q][nt], a, hb0[ks][nt], hb1[ks][nt]);
                            }
                        }
                } else {
                    mt0 = (b0 + b) * 2;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 v = lds128(stage + ((size_t)b * 2 + q) * 512 + lane * 16);
                        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nact) mma_16816(acc[q][nt], a, hb0[0][nt], hb1[0][nt]);
                    }
                }
                const int n0 = 32 * (mt0 >> 1) + 4 * g;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (nt < nact) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int col = col0 + nt * 8 + 2 * q4 + hf;
                            if (col < ui.n_e) {
                                const float w = c.tok_scale[col];
                                float4 v;
                                v.x = acc[0][nt][hf] * sd[0] * w;
                                v.y = acc[0][nt][2 + hf] * sd[1] * w;
                                v.z = acc[1][nt][hf] * sd[2] * w;
                                v.w = acc[1][nt][2 + hf] * sd[3] * w;
                                atomicAdd(reinterpret_cast<float4 *>(p.yout + (size_t)c.tok_row[col] * H + n0), v);
                            }
                        }
                    }
                }
            }
        }
    }
}

template <int MS4, int NT>
__global__ void __launch_bounds__(kThreads, 1) engine_kernel(const EngineParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(p.T, p.H, p.npad, p.nstages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + p.nstages;
    uint64_t *csync = empty + p.nstages;
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(csync, kConsumerWarps);
        misc[0] = 0;  // abort flag
        misc[1] = 0;  // last-block flag
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kConsumerWarps) {
        if (lane == 0) producer_loop(p, smem, L);
        return;
    }

    ConsumerCtx c;
    c.full = full;
    c.empty = empty;
    c.csync = csync;
    c.hdrs = reinterpret_cast<ChunkHeader *>(smem + L.hdrs);
    c.ring = smem + L.ring;
    c.tok_x = reinterpret_cast<int *>(smem + L.tok);
    c.tok_row = c.tok_x + kMaxT;
    c.tok_scale = reinterpret_cast<float *>(c.tok_row + kMaxT);
    c.gamma = c.tok_scale + kMaxT;
    c.abort_flag = reinterpret_cast<volatile int *>(misc);
    c.misc = misc;
    c.sc = reinterpret_cast<__half *>(smem + L.sc);
    c.red = reinterpret_cast<float *>(smem + L.red);
    c.hs = reinterpret_cast<__half *>(smem + L.hs);
    c.xs = reinterpret_cast<__half *>(smem + L.xs);
    c.xs_stride = L.xs_stride;
    c.csync_phase = 0;
    const int ctid = threadIdx.x;  // 0..255
    const int H = p.H;

    // stage activations [T][H] -> shared rows of H+8 halves
    {
        const int n16 = p.T * (H / 8);
        for (int idx = ctid; idx < n16; idx += kConsumerWarps * 32) {
            const int t = idx / (H / 8), h8 = idx - t * (H / 8);
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * H) + h8);
            *reinterpret_cast<uint4 *>(c.xs + (size_t)t * c.xs_stride + h8 * 8) = v;
        }
        for (int idx = ctid; idx < 64 * p.npad; idx += kConsumerWarps * 32) c.red[idx] = 0.f;
    }
    cons_sync(p, c);
    // shared-expert gate per token: gamma = 1 / (1 + exp(-x . w_sgate)), else 1
    if (p.shared && p.w_sgate) {
        for (int t = warp; t < p.T; t += kConsumerWarps) {
            float z = 0.f;
            for (int h = lane * 2; h < H; h += 64) {
                const float2 xv = __half22float2(*reinterpret_cast<const __half2 *>(c.xs + (size_t)t * c.xs_stride + h));
                const float2 wv = __half22float2(__ldg(reinterpret_cast<const __half2 *>(p.w_sgate + h)));
                z = fmaf(xv.x, wv.x, z);
                z = fmaf(xv.y, wv.y, z);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) c.gamma[t] = 1.0f / (1.0f + expf(-z));
        }
    } else {
        for (int t = ctid; t < p.T; t += kConsumerWarps * 32) c.gamma[t] = 1.0f;
    }
    cons_sync(p, c);

    const int n_sh = p.shared ? p.I_s / kF16S : 0;
    bool waited = false;
    UnitInfo ui{};
    ui.n_e = 0;
    uint32_t it = 0;
    const uint32_t it_cap = 1u << 30;
    while (it < it_cap) {
        const int st = it % p.nstages;
        if (!mbar_wait_bounded(&full[st], (it / p.nstages) & 1, c.abort_flag, &p.hdr->status, p.wait_budget_ns))
            break;
        const ChunkHeader h = c.hdrs[st];
        if (h.kind == HK_DONE) break;
        const int nb = h.nb_flags & 0xffff, flags = h.nb_flags >> 16;
        const uint8_t *stage = c.ring + (size_t)st * kChunk;
        if (flags & HF_UNIT_START) {
            cons_sync(p, c);
            if (h.unit >= n_sh && !waited) {
                griddep_wait();
                waited = true;
            }
            if (!decode_unit(p, h.unit, n_sh, ui)) ui.n_e = 0;
            if (warp == 0) {
                for (int i = lane; i < ui.n_e; i += 32) {
                    if (ui.is_shared) {
                        c.tok_x[i] = i;
                        c.tok_row[i] = i;
                        c.tok_scale[i] = p.mode == MODE_SORTED ? 1.0f : c.gamma[i];
                    } else {
                        const int pidx = __ldcg(p.offsets + ui.e) + i;
                        int s = __ldcg(p.sorted_slots + pidx);
                        s = (s >= 0 && s < p.T * p.k) ? s : 0;
                        const int t = s / p.k;
                        c.tok_x[i] = t;
                        if (p.mode == MODE_SORTED) {
                            c.tok_row[i] = pidx;
                            c.tok_scale[i] = 1.0f;
                        } else {
                            c.tok_row[i] = t;
                            c.tok_scale[i] = __ldcg(p.topk_w + s);
                        }
                    }
                }
            }
            if (h.kind == HK_SCALES) {
                const int n16 = (int)(w4_sc_bytes(H, ui.S) / 16);
                for (int idx = ctid; idx < n16; idx += kConsumerWarps * 32)
                    reinterpret_cast<uint4 *>(c.sc)[idx] = lds128(stage + idx * 16);
            }
            cons_sync(p, c);
        }
        if (ui.n_e > 0) {
            if (h.kind == HK_GU)
                process_gu<MS4, NT>(p, c, ui, stage, h.b0, nb);
            else if (h.kind == HK_DOWN)
                process_down<MS4, NT>(p, c, ui, stage, h.b0, nb);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (flags & HF_GU_LAST) {
            cons_sync(p, c);
            if (ui.n_e > 0) compute_h(p, c, ui);
            cons_sync(p, c);
        }
        ++it;
    }

    // completion ticket; the last block writes the fp16 output and resets
    cons_sync(p, c);
    if (ctid == 0) {
        __threadfence();
        const uint32_t t = atomicAdd(&p.hdr->done_ticket, 1u);
        misc[1] = (t == gridDim.x - 1);
    }
    cons_sync(p, c);
    if (misc[1]) {
        __threadfence();
        if (p.mode == MODE_LAYER) {
            const int n4 = p.T * H / 4;
            float4 *acc4 = reinterpret_cast<float4 *>(p.yout);
            for (int idx = ctid; idx < n4; idx += kConsumerWarps * 32) {
                const float4 v = __ldcg(acc4 + idx);
                __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
                uint2 o;
                o.x = h2_as_u32(lo);
                o.y = h2_as_u32(hi);
                reinterpret_cast<uint2 *>(p.out)[idx] = o;
                __stcg(acc4 + idx, make_float4(0.f, 0.f, 0.f, 0.f));
            }
        }
        if (ctid == 0) {
            p.hdr->work_counter = 0;
            p.hdr->done_ticket = 0;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------ launching --
template <int MS4, int NT>
static int launch_engine_t(const EngineParams &p0, cudaStream_t s, bool pdl) {
    EngineParams p = p0;
    const int sms = device_sm_count();
    if (sms <= 0) return SPX_ERR_CUDA;
    int nst = 12;
    SmemLayout L = smem_layout(p.T, p.H, p.npad, nst);
    while (nst > 2 && L.total > kSmemLimit) L = smem_layout(p.T, p.H, p.npad, --nst);
    if (L.total > kSmemLimit) return SPX_ERR_UNSUPPORTED;
    p.nstages = nst;
    static int configured[64][1] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return SPX_ERR_CUDA;
    if (!configured[dev][0]) {
        cudaError_t e = cudaFuncSetAttribute(engine_kernel<MS4, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemLimit);
        if (e != cudaSuccess) return record_launch(e);
        configured[dev][0] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, engine_kernel<MS4, NT>, p);
    return record_launch(e);
}

int launch_engine(const EngineParams &p, cudaStream_t s, bool pdl) {
    const int ms4 = p.routed_fmt == FMT_W4 ? p.S / 16 : 1;
    const bool wide = p.T > 8;
    if (ms4 == 2) return wide ? launch_engine_t<2, 3>(p, s, pdl) : launch_engine_t<2, 1>(p, s, pdl);
    return wide ? launch_engine_t<1, 3>(p, s, pdl) : launch_engine_t<1, 1>(p, s, pdl);
}

// fixed part of the engine's shared memory (for validation)
int engine_fits(int T, int H) {
    const int npad = 8 * ((T + 7) / 8);
    SmemLayout L = smem_layout(T, H, npad, 2);
    return L.total <= kSmemLimit;
}

}  // namespace spx
