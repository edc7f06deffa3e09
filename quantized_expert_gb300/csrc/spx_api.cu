// spx_api.cu -- C ABI entry points of libspx for the expert path: argument
// validation, workspace handling and launch sequencing.  Every numeric step
// runs in the kernels of spx_route.cu, spx_engine.cu and the combine kernel
// below; this file only checks arguments and enqueues launches.
#include "spx_internal.cuh"

#include <math.h>

namespace spx {

int device_sm_count() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int record_launch(cudaError_t e) {
    if (e == cudaSuccess) return SPX_OK;
    g_last_cuda_error = e;
    return SPX_ERR_CUDA;
}

// out[t][n] = fp16( sum_j w[t][j] * y_sorted[pos(t,j)][n] + acc[t][n] ); acc -> 0
__global__ void __launch_bounds__(256) combine_kernel(const float *y_sorted, const int32_t *sorted_slots,
                                                      const float *topk_w, float *acc, int T, int H, int k,
                                                      __half *out) {
    __shared__ int inv[kMaxSlots];
    const int n = T * k;
    for (int p = threadIdx.x; p < n; p += blockDim.x) {
        const int s = sorted_slots[p];
        if (s >= 0 && s < n) inv[s] = p;
    }
    __syncthreads();
    const int t = blockIdx.y;
    const int n4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T || n4 * 4 >= H) return;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (acc) {
        a = __ldcg(reinterpret_cast<const float4 *>(acc + (size_t)t * H) + n4);
        __stcg(reinterpret_cast<float4 *>(acc + (size_t)t * H) + n4, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const float w = topk_w[t * k + j];
        const float4 y = __ldg(reinterpret_cast<const float4 *>(y_sorted + (size_t)inv[t * k + j] * H) + n4);
        r.x = fmaf(w, y.x, r.x);
        r.y = fmaf(w, y.y, r.y);
        r.z = fmaf(w, y.z, r.z);
        r.w = fmaf(w, y.w, r.w);
    }
    __half2 lo = __floats2half2_rn(r.x + a.x, r.y + a.y), hi = __floats2half2_rn(r.z + a.z, r.w + a.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out + (size_t)t * H)[n4] = o;
}

}  // namespace spx

using namespace spx;

static const uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s per bounded wait

static bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

extern "C" const char *spx_status_string(int st) {
    switch (st) {
        case SPX_OK: return "ok";
        case SPX_ERR_INVALID_ARG: return "invalid argument";
        case SPX_ERR_UNSUPPORTED: return "unsupported shape";
        case SPX_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case SPX_ERR_CUDA: return "CUDA error";
        case SPX_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

extern "C" int spx_version(void) { return 106; }

extern "C" const char *spx_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

static size_t ws_scratch_base(int T, int H) { return ws_order_offset(T, H) + (size_t)kMaxE * 4; }

static size_t ws_size_core(int T, int H, int I, int E, int k, int I_s) {
    if (T < 1 || H < 1 || T > kMaxT || H > kMaxH || I < 0 || E < 1 || k < 1 || I_s < 0) return 0;
    const size_t base = ws_scratch_base(T, H);
    if (T > kDraftLaunchMaxT || I % 128 || I_s % 16) return base;  // only the draft launch has split-K scratch
    const int nact = E < T * k ? E : T * k;
    return draft_scratch_end(base, T, H, I, I_s, nact);
}
// The tensor-memory launches' scratch starts on the first 1024-byte boundary
// after the routing tables (it is never used together with the draft scratch).
static size_t ws_tc_offset(int T, int H) { return (ws_scratch_base(T, H) + 1023) / 1024 * 1024; }

extern "C" size_t spx_workspace_size_tc(int T, int H, int I, int E, int k, int I_s) {
    const size_t core = ws_size_core(T, H, I, E, k, I_s);
    if (!core || I < 64 || I % 64 || I_s % 64 || H % 128) return 0;
    const size_t tc = ws_tc_offset(T, H) + tc_scratch_bytes(T, H, I, E, k, I_s);
    return tc > core ? tc : core;
}

size_t spx::workspace_bytes(int T, int H, int I, int E, int k, int I_s, int launch) {
    if (launch == 1) return ws_size_core(T, H, I, E, k, I_s);
    if (launch == 2) return spx_workspace_size_tc(T, H, I, E, k, I_s);
    return spx_workspace_size(T, H, I, E, k, I_s);
}

extern "C" size_t spx_workspace_size(int T, int H, int I, int E, int k, int I_s) {
    const size_t core = ws_size_core(T, H, I, E, k, I_s);
    if (!core || !tc_preferred(T)) return core;
    const size_t tc = spx_workspace_size_tc(T, H, I, E, k, I_s);
    return tc > core ? tc : core;
}

static TokTable *ws_tables(void *ws, int T, int H) {
    return reinterpret_cast<TokTable *>(static_cast<uint8_t *>(ws) + ws_tables_offset(T, H));
}

extern "C" int spx_workspace_init(void *ws, size_t ws_bytes, spx_stream_t stream) {
    if (!ws || ws_bytes < sizeof(WsHeader)) return SPX_ERR_WORKSPACE;
    return record_launch(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int spx_workspace_status(const void *ws, int32_t *host_status, spx_stream_t stream) {
    if (!ws || !host_status) return SPX_ERR_INVALID_ARG;
    const WsHeader *h = static_cast<const WsHeader *>(ws);
    return record_launch(cudaMemcpyAsync(host_status, &h->status, sizeof(int32_t), cudaMemcpyDefault,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

static int check_expert_common(const uint16_t *x, int T, int H, int E, int I, int k, const int32_t *offsets,
                               const int32_t *sorted_slots, const int32_t *active, const int32_t *n_active,
                               void *ws, size_t ws_bytes, int fmt, int S, int I_s = 0, bool tc = false) {
    if (!x || !offsets || !sorted_slots || !active || !n_active) return SPX_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || E < 1 || k > E || H < 1 || I < 1) return SPX_ERR_INVALID_ARG;
    if (T > kMaxT || E > kMaxE || T * k > kMaxSlots || H % 128 || I % 128 || H > kMaxH) return SPX_ERR_UNSUPPORTED;
    if (fmt == 0 && S != 16 && S != 32) return SPX_ERR_UNSUPPORTED;
    if (!tc && !engine_fits(T, H, fmt, S)) return SPX_ERR_UNSUPPORTED;
    if (!al16(x)) return SPX_ERR_INVALID_ARG;
    const size_t need = workspace_bytes(T, H, I, E, k, I_s, tc ? 2 : 1);
    if (!ws || ws_bytes < need || !al16(ws)) return SPX_ERR_WORKSPACE;
    return SPX_OK;
}

static EngineParams base_params(const uint16_t *x, int T, int H, void *ws) {
    EngineParams p{};
    p.x = reinterpret_cast<const __half *>(x);
    p.T = T;
    p.H = H;
    p.hdr = static_cast<WsHeader *>(ws);
    p.npad = 8 * ((T + 7) / 8);
    p.wait_budget_ns = kWaitBudgetNs;
    return p;
}

extern "C" int spx_moe_draft_w4a16(const uint16_t *x, int T, const spx_w4_experts *w, int k, const int32_t *offsets,
                                   const int32_t *sorted_slots, const int32_t *active, const int32_t *n_active,
                                   float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream) {
    if (!w || !w->packed || !y_sorted) return SPX_ERR_INVALID_ARG;
    int st = check_expert_common(x, T, w->H, w->E, w->I, k, offsets, sorted_slots, active, n_active, ws, ws_bytes, 0,
                                 w->slice_cols);
    if (st) return st;
    if (!al16(w->packed) || !al16(y_sorted) || !al16(w->zeros)) return SPX_ERR_INVALID_ARG;
    const bool draft = draft_supported(T, w->H, w->I, w->slice_cols, 0, w->E, k);
    if (w->zeros && !draft && !engine_fits(T, w->H, kFmtW4Z, w->slice_cols)) return SPX_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EngineParams p = base_params(x, T, w->H, ws);
    p.routed = static_cast<const uint8_t *>(w->packed);
    p.w4_zeros = static_cast<const uint8_t *>(w->zeros);
    p.w4_sdown = reinterpret_cast<const __half *>(p.routed + w4_units_bytes(w->E, w->H, w->I, w->slice_cols));
    p.routed_fmt = 0;
    p.S = w->slice_cols;
    p.E = w->E;
    p.I = w->I;
    p.k = k;
    p.routed_enabled = 1;
    p.active = active;
    p.n_active = n_active;
    p.tables = ws_tables(ws, T, w->H);
    p.mode = 0;  // sorted rows
    p.yout = y_sorted;
    if (cudaMemsetAsync(y_sorted, 0, sizeof(float) * (size_t)T * k * w->H, s) != cudaSuccess) return SPX_ERR_CUDA;
    st = launch_tables(offsets, sorted_slots, active, n_active, T, k, w->E, ws_tables(ws, T, w->H), s);
    if (st) return st;
    if (draft) return launch_draft(p, nullptr, ws_scratch_base(T, w->H), false, s);
    return launch_engine(p, s, false);
}

static int gguf_fmt(const spx_gguf_experts *w) {
    switch (w->gate_up_type) {
    case SPX_GGUF_Q8_0: return kFmtQ8;
    case SPX_GGUF_Q2_K: return kFmtQ2K;
    case SPX_GGUF_Q4_K: return kFmtQ4K;
    default: return -1;
    }
}

extern "C" int spx_moe_draft_gguf(const uint16_t *x, int T, const spx_gguf_experts *w, int k, const int32_t *offsets,
                                   const int32_t *sorted_slots, const int32_t *active, const int32_t *n_active,
                                   float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream) {
    if (!w || !w->packed || !y_sorted) return SPX_ERR_INVALID_ARG;
    int st = check_expert_common(x, T, w->H, w->E, w->I, k, offsets, sorted_slots, active, n_active, ws, ws_bytes, 0,
                                 16);
    if (st) return st;
    if (!al16(w->packed) || !al16(y_sorted) || gguf_fmt(w) < 0) return SPX_ERR_INVALID_ARG;
    const bool draft = draft_supported(T, w->H, w->I, 16, 0, w->E, k, gguf_fmt(w) == kFmtQ2K || gguf_fmt(w) == kFmtQ4K);
    if (!draft && !engine_fits(T, w->H, gguf_fmt(w), 16)) return SPX_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EngineParams p = base_params(x, T, w->H, ws);
    p.routed = static_cast<const uint8_t *>(w->packed);
    p.routed_fmt = gguf_fmt(w);
    p.S = 16;
    p.E = w->E;
    p.I = w->I;
    p.k = k;
    p.routed_enabled = 1;
    p.active = active;
    p.n_active = n_active;
    p.tables = ws_tables(ws, T, w->H);
    p.mode = 0;  // sorted rows
    p.yout = y_sorted;
    if (cudaMemsetAsync(y_sorted, 0, sizeof(float) * (size_t)T * k * w->H, s) != cudaSuccess) return SPX_ERR_CUDA;
    st = launch_tables(offsets, sorted_slots, active, n_active, T, k, w->E, ws_tables(ws, T, w->H), s);
    if (st) return st;
    if (draft) return launch_draft(p, nullptr, ws_scratch_base(T, w->H), false, s);
    return launch_engine(p, s, false);
}

extern "C" int spx_moe_verify_fp16(const uint16_t *x, int T, const spx_f16_experts *w, int k, const int32_t *offsets,
                                   const int32_t *sorted_slots, const int32_t *active, const int32_t *n_active,
                                   float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream) {
    if (!w || !w->packed || !y_sorted) return SPX_ERR_INVALID_ARG;
    int st = check_expert_common(x, T, w->H, w->E, w->I, k, offsets, sorted_slots, active, n_active, ws, ws_bytes, 1,
                                 kF16S);
    if (st) return st;
    if (!al16(w->packed) || !al16(y_sorted)) return SPX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EngineParams p = base_params(x, T, w->H, ws);
    p.routed = static_cast<const uint8_t *>(w->packed);
    p.routed_fmt = 1;
    p.S = kF16S;
    p.E = w->E;
    p.I = w->I;
    p.k = k;
    p.routed_enabled = 1;
    p.active = active;
    p.n_active = n_active;
    p.tables = ws_tables(ws, T, w->H);
    p.mode = 0;
    p.yout = y_sorted;
    if (cudaMemsetAsync(y_sorted, 0, sizeof(float) * (size_t)T * k * w->H, s) != cudaSuccess) return SPX_ERR_CUDA;
    st = launch_tables(offsets, sorted_slots, active, n_active, T, k, w->E, ws_tables(ws, T, w->H), s);
    if (st) return st;
    return launch_engine(p, s, false);
}

extern "C" size_t spx_f16_tc_packed_bytes(int E, int H, int I) {
    if (E < 1 || H < 128 || I < 64 || H % 128 || I % 64 || H > kMaxH || E > kMaxE) return 0;
    return (size_t)E * tc_tiles(H, I) * 16384;
}

extern "C" int spx_f16_tc_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down, int E, int H,
                                 int I, void *tc_packed, spx_stream_t stream) {
    if (!w_gate || !w_up || !w_down || !tc_packed) return SPX_ERR_INVALID_ARG;
    if (!al16(w_gate) || !al16(w_up) || !al16(w_down) || !al16(tc_packed)) return SPX_ERR_INVALID_ARG;
    if (!spx_f16_tc_packed_bytes(E, H, I)) return SPX_ERR_UNSUPPORTED;
    return launch_tc_repack(w_gate, w_up, w_down, E, H, I, tc_packed, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int spx_shared_tc_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down, int H,
                                    int I_s, void *tc_packed, spx_stream_t stream) {
    return spx_f16_tc_repack(w_gate, w_up, w_down, 1, H, I_s, tc_packed, stream);
}

static int check_shared(const spx_shared *sh, int H) {
    if (!sh) return SPX_OK;
    if (!sh->packed || sh->H != H || sh->I_s < kF16S || sh->I_s % kF16S) return SPX_ERR_INVALID_ARG;
    if (!al16(sh->packed)) return SPX_ERR_INVALID_ARG;
    if (sh->w_sgate && !al16(sh->w_sgate)) return SPX_ERR_INVALID_ARG;
    return SPX_OK;
}

extern "C" int spx_combine(const float *y_sorted, const int32_t *sorted_slots, const float *topk_w, const uint16_t *x,
                           const spx_shared *shared, int T, int H, int k, uint16_t *out, void *ws, size_t ws_bytes,
                           spx_stream_t stream) {
    if (!y_sorted || !sorted_slots || !topk_w || !out) return SPX_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || H < 1) return SPX_ERR_INVALID_ARG;
    if (T > kMaxT || T * k > kMaxSlots || H % 128 || H > kMaxH) return SPX_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < spx_workspace_size(T, H, 0, 1, 1, 0) || !al16(ws)) return SPX_ERR_WORKSPACE;
    if (!al16(y_sorted) || (reinterpret_cast<uintptr_t>(out) & 7)) return SPX_ERR_INVALID_ARG;
    int st = check_shared(shared, H);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *acc = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kWsAccOffset);
    if (shared) {
        if (!x || !al16(x)) return SPX_ERR_INVALID_ARG;
        if (!engine_fits(T, H, 1, kF16S)) return SPX_ERR_UNSUPPORTED;
        EngineParams p = base_params(x, T, H, ws);
        p.routed_enabled = 0;
        p.routed_fmt = 1;
        p.S = kF16S;
        p.I = kF16S;
        p.E = 1;
        p.k = k;
        p.shared = static_cast<const uint8_t *>(shared->packed);
        p.w_sgate = reinterpret_cast<const __half *>(shared->w_sgate);
        p.I_s = shared->I_s;
        p.mode = 1;  // accumulate gamma * sh into acc
        p.yout = acc;
        st = launch_engine(p, s, false);
        if (st) return st;
    }
    dim3 grid((H / 4 + 255) / 256, T);
    combine_kernel<<<grid, 256, 0, s>>>(y_sorted, sorted_slots, topk_w, shared ? acc : nullptr, T, H, k,
                                        reinterpret_cast<__half *>(out));
    return record_launch(cudaGetLastError());
}

extern "C" int spx_moe_layer(const spx_layer_args *a, spx_stream_t stream) {
    return moe_layer(a, reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

int spx::moe_layer(const spx_layer_args *a, cudaStream_t s, void *clear, size_t clear_bytes) {
    if (!a) return SPX_ERR_INVALID_ARG;
    const int T = a->T, H = a->H, E = a->E, k = a->k;
    int st = route_validate(a->x, a->w_router, a->logits, T, H, E, k, a->topk_ids, a->topk_w);
    if (st) return st;
    if (!a->x || !a->counts || !a->offsets || !a->sorted_slots || !a->active || !a->n_active || !a->out)
        return SPX_ERR_INVALID_ARG;
    if (a->mode != 0 && a->mode != 1) return SPX_ERR_INVALID_ARG;
    if (a->elb && (a->layer < 0 || a->layer >= a->L)) return SPX_ERR_INVALID_ARG;
    int I = 0;
    const uint8_t *routed = nullptr;
    int S = kF16S;
    const bool gguf = a->mode == 0 && a->gguf;
    if (gguf) {
        if (a->w4 || !a->gguf->packed || a->gguf->E != E || a->gguf->H != H) return SPX_ERR_INVALID_ARG;
        if (!al16(a->gguf->packed) || gguf_fmt(a->gguf) < 0) return SPX_ERR_INVALID_ARG;
        I = a->gguf->I;
        S = 16;
        routed = static_cast<const uint8_t *>(a->gguf->packed);
    } else if (a->mode == 0) {
        if (!a->w4 || !a->w4->packed || a->w4->E != E || a->w4->H != H) return SPX_ERR_INVALID_ARG;
        if (!al16(a->w4->packed) || !al16(a->w4->zeros)) return SPX_ERR_INVALID_ARG;
        I = a->w4->I;
        S = a->w4->slice_cols;
        routed = static_cast<const uint8_t *>(a->w4->packed);
    } else {
        if (!a->f16 || !a->f16->packed || a->f16->E != E || a->f16->H != H) return SPX_ERR_INVALID_ARG;
        if (!al16(a->f16->packed)) return SPX_ERR_INVALID_ARG;
        I = a->f16->I;
        routed = static_cast<const uint8_t *>(a->f16->packed);
    }
    const int I_s = a->shared ? a->shared->I_s : 0;
    const bool cache_aware = a->resident || a->ready;
    // verify: the tensor-memory launches (canonical FP16 matrices) or the expert launch
    bool use_tc = false;
    if (a->mode == 1) {
        if (a->verify_launch < 0 || a->verify_launch > 2) return SPX_ERR_INVALID_ARG;
        const spx_shared *sh = a->shared;
        if (!al16(a->f16->tc_packed) || (sh && !al16(sh->tc_packed))) return SPX_ERR_INVALID_ARG;
        const bool canon = a->f16->tc_packed && (!sh || sh->tc_packed) && I % 64 == 0 && I_s % 64 == 0;
        if (a->verify_launch == 2) {
            if (!canon || cache_aware) return SPX_ERR_UNSUPPORTED;
            use_tc = true;
        } else if (a->verify_launch == 0) {
            use_tc = canon && !cache_aware && tc_preferred(T);
        }
    }
    st = check_expert_common(a->x, T, H, E, I, k, a->offsets, a->sorted_slots, a->active, a->n_active, a->ws,
                             a->ws_bytes, a->mode == 0 ? 0 : 1, S, I_s, use_tc);
    if (st) return st;
    st = check_shared(a->shared, H);
    if (st) return st;
    if (reinterpret_cast<uintptr_t>(a->out) & 7) return SPX_ERR_INVALID_ARG;
    const bool timed = a->ev_experts_begin || a->ev_experts_end;
    const uint64_t budget = a->wait_budget_ns ? a->wait_budget_ns : kWaitBudgetNs;

    const bool zeros = a->mode == 0 && !gguf && a->w4->zeros;
    const bool kq = gguf && (gguf_fmt(a->gguf) == kFmtQ2K || gguf_fmt(a->gguf) == kFmtQ4K);
    const bool via_draft = !cache_aware && draft_supported(T, H, I, S, I_s, E, k, kq);
    if (gguf && !via_draft && !engine_fits(T, H, gguf_fmt(a->gguf), 16)) return SPX_ERR_UNSUPPORTED;
    if (zeros && !via_draft && !engine_fits(T, H, kFmtW4Z, S)) return SPX_ERR_UNSUPPORTED;
    // the tensor-memory launches' parameters (their tensor maps checked) before anything is enqueued
    TcPlan tc_storage;
    TcPlan *tc = nullptr;
    if (use_tc) {
        TcArgs t{};
        t.x = reinterpret_cast<const __half *>(a->x);
        t.T = T;
        t.H = H;
        t.E = E;
        t.I = I;
        t.k = k;
        t.I_s = I_s;
        t.routed_tc = a->f16->tc_packed;
        if (a->shared) {
            t.shared_tc = a->shared->tc_packed;
            t.w_sgate = reinterpret_cast<const __half *>(a->shared->w_sgate);
        }
        t.active = a->active;
        t.n_active = a->n_active;
        t.tables = ws_tables(a->ws, T, H);
        t.scratch = static_cast<uint8_t *>(a->ws) + ws_tc_offset(T, H);
        t.acc = reinterpret_cast<float *>(static_cast<uint8_t *>(a->ws) + kWsAccOffset);
        t.out = reinterpret_cast<__half *>(a->out);
        t.hdr = static_cast<WsHeader *>(a->ws);
        t.wait_budget_ns = budget;
        st = tc_plan(t, &tc_storage);
        if (st) return st;
        tc = &tc_storage;
    }
    // every check has passed: only now may the caller's scratch be cleared
    if (clear) {
        const cudaError_t ce = cudaMemsetAsync(clear, 0, clear_bytes, s);
        if (ce != cudaSuccess) return record_launch(ce);
    }
    if (a->mode == 0 && !cache_aware && via_draft) {
        // Draft layer: the draft launch routes its few tokens itself (no
        // routing launch before it); with a router weight a small launch
        // computes the logits first and the draft launch overlaps it.
        if (a->w_router) {
            st = launch_router_logits(reinterpret_cast<const __half *>(a->x),
                                      reinterpret_cast<const __half *>(a->w_router), T, H, E, a->logits, s, !timed);
            if (st) return st;
        }
        DraftRouting rt{};
        rt.logits = a->logits;
        rt.renorm = a->renorm;
        rt.topk_ids = a->topk_ids;
        rt.topk_w = a->topk_w;
        rt.elb = a->elb;
        rt.layer = a->layer;
        rt.counts = a->counts;
        rt.offsets = a->offsets;
        rt.sorted_slots = a->sorted_slots;
        rt.active = a->active;
        rt.n_active = a->n_active;
        EngineParams p = base_params(a->x, T, H, a->ws);
        p.routed = routed;
        p.routed_fmt = gguf ? gguf_fmt(a->gguf) : 0;
        p.w4_zeros = gguf ? nullptr : static_cast<const uint8_t *>(a->w4->zeros);
        p.S = S;
        p.E = E;
        p.I = I;
        p.k = k;
        if (a->shared) {
            p.shared = static_cast<const uint8_t *>(a->shared->packed);
            p.w_sgate = reinterpret_cast<const __half *>(a->shared->w_sgate);
            p.I_s = a->shared->I_s;
        }
        p.mode = 2;
        p.yout = reinterpret_cast<float *>(static_cast<uint8_t *>(a->ws) + kWsAccOffset);
        p.out = reinterpret_cast<__half *>(a->out);
        p.wait_budget_ns = budget;
        if (a->ev_experts_begin && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_begin), s) != cudaSuccess)
            return SPX_ERR_CUDA;
        st = launch_draft(p, &rt, ws_scratch_base(T, H), !timed, s);
        if (st) return st;
        if (a->ev_experts_end && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_end), s) != cudaSuccess)
            return SPX_ERR_CUDA;
        return SPX_OK;
    }

    RouteParams rp{};
    rp.x = reinterpret_cast<const __half *>(a->x);
    rp.w_router = reinterpret_cast<const __half *>(a->w_router);
    rp.logits = a->logits;
    rp.T = T;
    rp.H = H;
    rp.E = E;
    rp.k = k;
    rp.renorm = a->renorm;
    rp.topk_ids = a->topk_ids;
    rp.topk_w = a->topk_w;
    rp.elb = a->elb;
    rp.layer = a->layer;
    rp.counts = a->counts;
    rp.offsets = a->offsets;
    rp.sorted_slots = a->sorted_slots;
    rp.active = a->active;
    rp.n_active = a->n_active;
    rp.tables = ws_tables(a->ws, T, H);
    if (a->resident) {
        rp.resident = a->resident;
        rp.order = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(a->ws) + ws_order_offset(T, H));
    }
    rp.hdr = static_cast<WsHeader *>(a->ws);
    st = launch_route(rp, s, !timed);
    if (st) return st;

    if (use_tc) {
        if (a->ev_experts_begin && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_begin), s) != cudaSuccess)
            return SPX_ERR_CUDA;
        st = launch_tc_plan(*tc, s, !timed);
        if (st) return st;
        if (a->ev_experts_end && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_end), s) != cudaSuccess)
            return SPX_ERR_CUDA;
        return SPX_OK;
    }

    EngineParams p = base_params(a->x, T, H, a->ws);
    p.routed = routed;
    p.routed_fmt = gguf ? gguf_fmt(a->gguf) : a->mode == 0 ? 0 : 1;
    p.w4_zeros = zeros ? static_cast<const uint8_t *>(a->w4->zeros) : nullptr;
    p.S = S;
    if (a->mode == 0 && !gguf) p.w4_sdown = reinterpret_cast<const __half *>(routed + w4_units_bytes(E, H, I, S));
    p.E = E;
    p.I = I;
    p.k = k;
    p.routed_enabled = 1;
    p.active = a->active;
    p.n_active = a->n_active;
    p.order = rp.order;
    p.ready = a->ready;
    p.wait_budget_ns = budget;
    p.tables = ws_tables(a->ws, T, H);
    if (a->shared) {
        p.shared = static_cast<const uint8_t *>(a->shared->packed);
        p.w_sgate = reinterpret_cast<const __half *>(a->shared->w_sgate);
        p.I_s = a->shared->I_s;
    }
    p.mode = 2;  // layer: weighted accumulate, last block writes out
    p.yout = reinterpret_cast<float *>(static_cast<uint8_t *>(a->ws) + kWsAccOffset);
    p.out = reinterpret_cast<__half *>(a->out);
    if (a->ev_experts_begin && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_begin), s) != cudaSuccess)
        return SPX_ERR_CUDA;
    st = launch_engine(p, s, !timed);
    if (st) return st;
    if (a->ev_experts_end && cudaEventRecord(static_cast<cudaEvent_t>(a->ev_experts_end), s) != cudaSuccess)
        return SPX_ERR_CUDA;
    return SPX_OK;
}
