// spx_route.cu -- router product, softmax + top-k, Expert Lookahead Buffer
// counters and the counting-sort gather, as one small launch.
//
// Method (ai.info summary of the Specter paper, Key Contributions 2-4 and
// "Methodology in Plain English"; richland.au post, "What shipped"): the draft
// shares the target's FP16 router; GPU-side counters tally per layer how often
// each expert is selected by draft tokens; tokens are gathered by expert so
// each expert's work is dispatched once.
//
// Layout of the launch: when a router weight is given, one block per expert
// row computes that row's logits for every token (fp32 accumulate) and the
// last block to finish (completion ticket in the workspace, no spin) selects;
// otherwise a single block selects from the given logits.  Selection: one
// warp per token (rank of each expert in the order value descending, index
// ascending; softmax with expf), then the counting sort by one block.
#include "spx_internal.cuh"
#include "spx_routing.cuh"

#include <math.h>

namespace spx {


__device__ __forceinline__ float dot8_h(uint4 a, uint4 b, float acc) {
    const __half2 *pa = reinterpret_cast<const __half2 *>(&a);
    const __half2 *pb = reinterpret_cast<const __half2 *>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 fa = __half22float2(pa[i]);
        float2 fb = __half22float2(pb[i]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
    }
    return acc;
}

// logits[t][e] of expert row e = blockIdx.x for every token t: a thread
// holds every H/8 / blockDim-th uint4 of the row, its loads of the row issued
// together; tokens in passes of 8, fp32 accumulate, warp then block
// reduction.  Any block size that is a multiple of 32, at most 1024.
__device__ void router_row_block(const __half *x, const __half *wr, int T, int H, int E, float *logits) {
    __shared__ float red[32][8];
    const int e = blockIdx.x, nthr = blockDim.x, nw = nthr >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4 *w4 = reinterpret_cast<const uint4 *>(wr + (size_t)e * H);
    const uint4 *x4 = reinterpret_cast<const uint4 *>(x);
    const int H8 = H / 8;
    for (int t0 = 0; t0 < T; t0 += 8) {
        float acc[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = 0.f;
#pragma unroll 4
        for (int h8 = threadIdx.x; h8 < H8; h8 += nthr) {
            const uint4 w = __ldg(w4 + h8);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (t0 + t < T) acc[t] = dot8_h(__ldg(x4 + (size_t)(t0 + t) * H8 + h8), w, acc[t]);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][t] = v;
        }
        __syncthreads();
        if (threadIdx.x < 8 && t0 + (int)threadIdx.x < T) {
            float v = 0.f;
            for (int w = 0; w < nw; ++w) v += red[w][threadIdx.x];
            logits[(size_t)(t0 + threadIdx.x) * E + e] = v;
        }
        __syncthreads();
    }
}

// Counting sort of the T*k slots held in s_ids (shared) into the caller's
// gather arrays.  Whole block participates.
__device__ void gather_block(const int32_t *s_ids, int n, int E, int32_t *counts, int32_t *offsets,
                             int32_t *sorted_slots, int32_t *active, int32_t *n_active, int k = 1,
                             const float *s_w = nullptr, TokTable *tables = nullptr,
                             const uint8_t *resident = nullptr, int32_t *order = nullptr) {
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_off[kMaxE + 1];
    __shared__ int s_act[kMaxE];
    __shared__ int s_na;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int s = tid; s < n; s += blockDim.x) atomicAdd(&s_cnt[s_ids[s]], 1);
    __syncthreads();
    if (tid < 32) {
        // exclusive scans of counts and of (count > 0); each lane owns a run of 8
        const int lane = tid;
        int c[8], f[8];
        int sc = 0, sf = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int e = lane * 8 + i;
            c[i] = e < E ? s_cnt[e] : 0;
            f[i] = c[i] > 0;
            sc += c[i];
            sf += f[i];
        }
        int ic = sc, jf = sf;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int a = __shfl_up_sync(0xffffffffu, ic, o);
            int b = __shfl_up_sync(0xffffffffu, jf, o);
            if (lane >= o) {
                ic += a;
                jf += b;
            }
        }
        int run = ic - sc, runf = jf - sf;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int e = lane * 8 + i;
            if (e < E) {
                s_off[e] = run;
                if (f[i]) s_act[runf] = e;
            }
            run += c[i];
            runf += f[i];
        }
        if (lane == 31) {
            s_off[E] = ic;
            *n_active = jf;
            s_na = jf;
            for (int a = jf; a < E; ++a) s_act[a] = -1;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        counts[e] = s_cnt[e];
        offsets[e] = s_off[e];
        active[e] = s_act[e];
    }
    if (tid == 0) offsets[E] = s_off[E];
    // stable placement: rank of slot s among earlier slots of the same expert
    for (int s = tid; s < n; s += blockDim.x) {
        const int e = s_ids[s];
        int rank = 0;
        for (int s2 = 0; s2 < s; ++s2) rank += (s_ids[s2] == e);
        sorted_slots[s_off[e] + rank] = s;
        if (tables) {
            // token table of expert e, entry rank: token s/k, output row s/k, gate weight
            TokEntry te;
            te.tok = s / k;
            te.row = s / k;
            te.scale = s_w[s];
            te.pad = 0;
            tables[e].e[rank] = te;
        }
    }
    if (tables)
        for (int e = tid; e < E; e += blockDim.x)
            if (s_cnt[e] > 0) tables[e].n = s_cnt[e];
    if (order) {
        // the expert launch's queue: resident experts first, then the others,
        // each in ascending expert order (the active list's order)
        __shared__ unsigned char s_res[kMaxE];
        const int na = s_na;
        for (int a = tid; a < na; a += blockDim.x) s_res[a] = resident[s_act[a]] != 0;
        __syncthreads();
        for (int a = tid; a < na; a += blockDim.x) {
            const int r = s_res[a];
            int before = 0, nres = 0;
            for (int a2 = 0; a2 < na; ++a2) {
                nres += s_res[a2];
                before += (a2 < a && s_res[a2] == r) ? 1 : 0;
            }
            order[r ? before : nres + before] = s_act[a];
        }
    }
}

// Softmax, top-k, weights, counters and gather; one block.
__device__ void select_block(const RouteParams &p) {
    __shared__ int32_t s_ids[kMaxSlots];
    __shared__ float s_pw[kMaxSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int t = warp; t < p.T; t += wpb) {
        const float *lg = p.logits + (size_t)t * p.E;
        select_token([&](int e) { return __ldcg(lg + e); }, p.E, p.k, p.renorm, lane, s_ids + t * p.k,
                     s_pw + t * p.k, nullptr);
        if (lane == 0)
            for (int r = 0; r < p.k; ++r) {
                const int be = s_ids[t * p.k + r];
                p.topk_ids[(size_t)t * p.k + r] = be;
                p.topk_w[(size_t)t * p.k + r] = s_pw[t * p.k + r];
                if (p.elb) atomicAdd(p.elb + (size_t)p.layer * p.E + be, 1u);
            }
    }
    __syncthreads();
    if (p.counts)
        gather_block(s_ids, p.T * p.k, p.E, p.counts, p.offsets, p.sorted_slots, p.active, p.n_active, p.k, s_pw,
                     p.tables, p.resident, p.order);
}

__global__ void __launch_bounds__(1024) route_kernel(const RouteParams p) {
    // Let a programmatically dependent expert launch start its routing-
    // independent work (shared expert) while this one runs; this one reads
    // nothing before the launch it follows has completed.
    griddep_launch_dependents();
    griddep_wait();
    if (p.w_router) {
        router_row_block(p.x, p.w_router, p.T, p.H, p.E, p.logits);
        __shared__ int s_last;
        if (threadIdx.x == 0) {
            __threadfence();
            s_last = atomicAdd(&p.hdr->route_ticket, 1u) == gridDim.x - 1;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (threadIdx.x == 0) p.hdr->route_ticket = 0;
    }
    select_block(p);
}

// Router product for the draft layer call (T <= 5): one block per expert row.
// A dependent launch may start at once and waits for the logits with
// griddepcontrol.wait.
__global__ void __launch_bounds__(256) router_logits_kernel(const __half *x, const __half *wr, int T, int H, int E,
                                                            float *logits) {
    griddep_launch_dependents();
    griddep_wait();
    router_row_block(x, wr, T, H, E, logits);
}

// pdl: the launch may begin while the preceding one on the stream finishes
// (programmatic dependent launch; the kernel waits for it before reading).
static cudaLaunchConfig_t small_launch(dim3 grid, dim3 block, cudaStream_t s, bool pdl, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

int launch_router_logits(const __half *x, const __half *wr, int T, int H, int E, float *logits, cudaStream_t s,
                         bool pdl) {
    if (T < 1 || T > 8) return SPX_ERR_UNSUPPORTED;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = small_launch(dim3(E), dim3(256), s, pdl, attr);
    return record_launch(cudaLaunchKernelEx(&cfg, router_logits_kernel, x, wr, T, H, E, logits));
}

__global__ void __launch_bounds__(256) elb_kernel(uint32_t *elb, int E, int layer, const int32_t *ids, int n) {
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < n; s += gridDim.x * blockDim.x) {
        const int e = ids[s];
        if (e >= 0 && e < E) atomicAdd(elb + (size_t)layer * E + e, 1u);
    }
}

__global__ void __launch_bounds__(256) gather_kernel(const int32_t *ids, int n, int E, int32_t *counts,
                                                      int32_t *offsets, int32_t *sorted_slots, int32_t *active,
                                                      int32_t *n_active) {
    __shared__ int32_t s_ids[kMaxSlots];
    for (int s = threadIdx.x; s < n; s += blockDim.x) {
        const int e = ids[s];
        s_ids[s] = (e >= 0 && e < E) ? e : 0;
    }
    __syncthreads();
    gather_block(s_ids, n, E, counts, offsets, sorted_slots, active, n_active);
}

// ----------------------------------------------------------- launchers --
static int check_route_shape(int T, int H, int E, int k) {
    if (T < 1 || E < 1 || k < 1 || H < 0) return SPX_ERR_INVALID_ARG;
    if (k > E) return SPX_ERR_INVALID_ARG;
    if (T > kMaxT || E > kMaxE || T * k > kMaxSlots) return SPX_ERR_UNSUPPORTED;
    return SPX_OK;
}

// One warp per token in the selecting block (at least 8 warps, at most 32);
// with a router weight one block per expert row, the last to finish selects.
int launch_route(const RouteParams &p, cudaStream_t s, bool pdl) {
    const int grid = p.w_router ? p.E : 1;
    const int threads = 32 * (p.T < 8 ? 8 : (p.T > 32 ? 32 : p.T));
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = small_launch(dim3(grid), dim3(threads), s, pdl, attr);
    return record_launch(cudaLaunchKernelEx(&cfg, route_kernel, p));
}

int route_preload() {
    cudaFuncAttributes fa;
    int st = record_launch(cudaFuncGetAttributes(&fa, route_kernel));
    if (!st) st = record_launch(cudaFuncGetAttributes(&fa, router_logits_kernel));
    return st;
}

int route_validate(const uint16_t *x, const uint16_t *w_router, const float *logits, int T, int H, int E, int k,
                   const int32_t *ids, const float *w) {
    int st = check_route_shape(T, H, E, k);
    if (st) return st;
    if (!logits || !ids || !w) return SPX_ERR_INVALID_ARG;
    if (w_router) {
        if (!x) return SPX_ERR_INVALID_ARG;
        if (H % 128 || H > kMaxH || H < 128) return SPX_ERR_UNSUPPORTED;
        if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15) return SPX_ERR_INVALID_ARG;
    }
    return SPX_OK;
}

}  // namespace spx

using namespace spx;

extern "C" int spx_route_topk(const uint16_t *x, const uint16_t *w_router, float *logits, int T, int H, int E,
                              int k, int renorm, int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                              spx_stream_t stream) {
    int st = route_validate(x, w_router, logits, T, H, E, k, topk_ids, topk_w);
    if (st) return st;
    if (w_router && (!ws || ws_bytes < sizeof(WsHeader))) return SPX_ERR_WORKSPACE;
    RouteParams p{};
    p.x = reinterpret_cast<const __half *>(x);
    p.w_router = reinterpret_cast<const __half *>(w_router);
    p.logits = logits;
    p.T = T;
    p.H = H;
    p.E = E;
    p.k = k;
    p.renorm = renorm;
    p.topk_ids = topk_ids;
    p.topk_w = topk_w;
    p.hdr = reinterpret_cast<WsHeader *>(ws);
    return launch_route(p, reinterpret_cast<cudaStream_t>(stream), false);
}

extern "C" int spx_elb_accumulate(uint32_t *elb, int L, int E, int layer, const int32_t *topk_ids, int T, int k,
                                  spx_stream_t stream) {
    if (!elb || !topk_ids || L < 1 || E < 1 || T < 1 || k < 1 || layer < 0 || layer >= L || k > E)
        return SPX_ERR_INVALID_ARG;
    if (E > kMaxE || T > kMaxT || T * k > kMaxSlots) return SPX_ERR_UNSUPPORTED;
    elb_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(elb, E, layer, topk_ids, T * k);
    return record_launch(cudaGetLastError());
}

extern "C" int spx_elb_read(const uint32_t *elb, int L, int E, uint32_t *dst, spx_stream_t stream) {
    if (!elb || !dst || L < 1 || E < 1) return SPX_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(dst, elb, sizeof(uint32_t) * (size_t)L * E, cudaMemcpyDefault,
                                    reinterpret_cast<cudaStream_t>(stream));
    return record_launch(e);
}

extern "C" int spx_elb_reset(uint32_t *elb, int L, int E, spx_stream_t stream) {
    if (!elb || L < 1 || E < 1) return SPX_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(elb, 0, sizeof(uint32_t) * (size_t)L * E, reinterpret_cast<cudaStream_t>(stream));
    return record_launch(e);
}

extern "C" int spx_gather_by_expert(const int32_t *topk_ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                                    int32_t *sorted_slots, int32_t *active, int32_t *n_active, spx_stream_t stream) {
    if (!topk_ids || !counts || !offsets || !sorted_slots || !active || !n_active) return SPX_ERR_INVALID_ARG;
    int st = check_route_shape(T, 0, E, k);
    if (st) return st;
    gather_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(topk_ids, T * k, E, counts, offsets,
                                                                         sorted_slots, active, n_active);
    return record_launch(cudaGetLastError());
}
