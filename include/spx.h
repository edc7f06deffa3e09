/*
 * spx.h -- C ABI of libspx, the GB300 (sm_103a) per-layer MoE expert path of
 * Specter's Streamlined Execution Engine, for one decoding request.
 *
 * Sources, cited by page title and section:
 *  [P1] ai.info summary, "Specter: Fast MoE Inference via Quantization-Enabled
 *       Multi-Step Speculative Offloading": Key Contributions 2 (FP16 gates and
 *       shared experts, INT4 routed experts), 3 (Expert Lookahead Buffer: GPU-
 *       resident, layer-indexed expert-activation counters), 4 (fused multi-
 *       expert INT4 draft kernel that gathers tokens by expert in one launch;
 *       expert-wise verification reordering); "Methodology in Plain English";
 *       Main Findings (routing fidelity of drafts quantised by GPTQ, AWQ and
 *       GGUF at Q2, Q4 and Q8: the other draft formats below).
 *  [P2] richland.au, "Specter previews expert routing with an INT4 copy of the
 *       model itself", section "What shipped": GPTQ INT4 with group size 128,
 *       routers and shared experts reuse the target's FP16 tensors, W4A16
 *       kernels that dequantise INT4 tiles and compute in FP16.
 *
 * Conventions (all entry points):
 *  - fp16 values are passed as binary16 bit patterns (uint16_t); fp32 as float.
 *  - Every pointer is caller-owned device memory unless stated otherwise; the
 *    library allocates nothing and never synchronises.  Every call is
 *    asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Arguments are validated before any launch.  Return value: SPX_OK, or a
 *    negative spx_status; on error nothing was enqueued.  Launch failures are
 *    reported as SPX_ERR_CUDA (from cudaGetLastError).
 *  - Supported shapes: 1 <= T <= 64 tokens, 1 <= k <= E <= 256, T*k <= 512,
 *    H and I multiples of 128, H <= 8192.  Anything else: SPX_ERR_UNSUPPORTED.
 *  - Device pointers passed to the expert calls must be 16-byte aligned.
 *  - The library holds no state between calls: the counter table and the
 *    workspace are the caller's buffers.  One workspace must not be used by
 *    two calls that can run concurrently (e.g. on two streams).
 *  - The expert launches run one block per SM and some of their blocks wait
 *    for others (finished work, intermediate results); every such wait is
 *    bounded: if other work keeps SMs from this launch for longer than the
 *    bound, the call's status word becomes SPX_ERR_TIMEOUT.
 */
#ifndef SPX_H
#define SPX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPX_API __attribute__((visibility("default")))
#else
#define SPX_API
#endif

typedef struct CUstream_st *spx_stream_t; /* same type as cudaStream_t */

typedef enum {
    SPX_OK = 0,
    SPX_ERR_INVALID_ARG = -1, /* null pointer, negative size, k > E, ... */
    SPX_ERR_UNSUPPORTED = -2, /* shape outside the supported range */
    SPX_ERR_WORKSPACE = -3,   /* workspace missing, too small or misaligned */
    SPX_ERR_CUDA = -4,        /* a CUDA call or kernel launch failed */
    SPX_ERR_TIMEOUT = -5      /* a bounded device-side wait gave up (status word) */
} spx_status;

/* Static text for a status code (never NULL). */
SPX_API const char *spx_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
SPX_API int spx_version(void);

/* Text of the last CUDA error this thread's calls turned into SPX_ERR_CUDA
 * ("no error" if none); static storage, never NULL. */
SPX_API const char *spx_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Router: logits, softmax, top-k   [P1 Key Contributions 2; P2 What shipped] */
/* ------------------------------------------------------------------------ */
/* logits: [T][E] fp32.  If w_router != NULL (fp16 [E][H]) the call computes
 *   logits[t][e] = sum_h x[t][h] * w_router[e][h] (fp32 accumulate) and writes
 *   them; otherwise logits is read as given and x may be NULL.
 * Selection: the k largest fp32 logits per token, ties to the lower expert
 *   index, in descending order -> topk_ids [T][k] (int32).
 * Weights: p = softmax over all E experts; topk_w[t][j] = p[id] (renorm == 0)
 *   or p[id] / sum of the k selected p (renorm != 0) -> [T][k] fp32.
 * ws: workspace of spx_workspace_size(T, H, 0, E, k, 0) bytes or more (holds
 *   the completion counter of the multi-block router product). */
SPX_API int spx_route_topk(const uint16_t *x, const uint16_t *w_router, float *logits,
                   int T, int H, int E, int k, int renorm,
                   int32_t *topk_ids, float *topk_w,
                   void *ws, size_t ws_bytes, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert Lookahead Buffer counters  [P1 Key Contributions 3; Methodology]   */
/* ------------------------------------------------------------------------ */
/* elb: uint32 [L][E], layer-indexed expert-activation counters.
 * accumulate: elb[layer][topk_ids[t][j]] += 1 for every t < T, j < k
 *   (so each call adds exactly T*k to the layer's row). */
SPX_API int spx_elb_accumulate(uint32_t *elb, int L, int E, int layer,
                       const int32_t *topk_ids, int T, int k, spx_stream_t stream);
/* read: asynchronous, non-destructive snapshot of all L*E counters into dst,
 *   which may be device memory or page-locked host memory. */
SPX_API int spx_elb_read(const uint32_t *elb, int L, int E, uint32_t *dst, spx_stream_t stream);
/* reset: all L*E counters to zero. */
SPX_API int spx_elb_reset(uint32_t *elb, int L, int E, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Layer-Aware Prefetch Planner  [P1 Key Contributions 3 (counter snapshots  */
/* feed a planner with Cold Start, Prefetch Overlap and Final Cleanup phases  */
/* and adaptively sized draft chunks); Methodology (chunks sized so compute  */
/* roughly matches transfer time on a parallel stream); P2 What shipped (a   */
/* compact prefetch plan at chunk boundaries)]                                */
/* ------------------------------------------------------------------------ */
/* The pages name the phases and the sizing goal only; the rule below is this
 * library's reading.  One call per draft-chunk boundary of a speculation cycle
 * of K draft steps (host code; all pointers host memory):
 *  phase: SPX_PLAN_COLD_START when steps_done == 0, SPX_PLAN_PREFETCH_OVERLAP
 *    when 0 < steps_done < K, SPX_PLAN_FINAL_CLEANUP when steps_done == K.
 *  demand of layer l: experts e with elb[l][e] > 0 (a snapshot of the counters
 *    after steps_done draft steps, e.g. from spx_elb_read) and cached[l][e] == 0,
 *    most counted first, ties to the lower expert index.
 *  actions, layers ascending (the order the verify pass needs them in): each
 *    demanded expert is loaded; when the layer already caches cfg->capacity
 *    experts, the lowest-index cached expert with a zero count is evicted
 *    first; when every cached expert has a nonzero count, the layer's remaining
 *    demand is left to the verify pass.  cached[][] (in/out) is updated.
 *    actions[3*i .. 3*i+2] = {layer, expert, SPX_PLAN_LOAD or SPX_PLAN_EVICT}.
 *  next_chunk: draft steps to run before the next call = ceil(loads *
 *    copy_us / step_us) clamped to [min_chunk, K - steps_done] (cold start with
 *    no load: min_chunk; final cleanup: 0).
 * max_actions must be at least twice the number of demanded experts (2*L*E is
 * always enough); otherwise SPX_ERR_INVALID_ARG and nothing is changed. */
enum { SPX_PLAN_COLD_START = 0, SPX_PLAN_PREFETCH_OVERLAP = 1, SPX_PLAN_FINAL_CLEANUP = 2 };
enum { SPX_PLAN_EVICT = 0, SPX_PLAN_LOAD = 1 };
typedef struct {
    int L, E, K;       /* layers, experts per layer, draft steps per cycle */
    int capacity;      /* experts of one layer the device holds at once (1..E) */
    int min_chunk;     /* least draft steps per chunk (>= 1) */
    double step_us;    /* device time of one draft step through all L layers (> 0) */
    double copy_us;    /* host-to-device time of one expert's weights (>= 0) */
} spx_plan_cfg;
SPX_API int spx_plan_prefetch(const spx_plan_cfg *cfg, const uint32_t *elb, int steps_done, uint8_t *cached,
                              int32_t *actions, int max_actions, int *n_actions, int *next_chunk, int *phase);
/* Executor of a plan on `stream` (a stream parallel to the compute stream):
 * per SPX_PLAN_LOAD, one cudaMemcpyAsync of expert e's expert_bytes from
 * host_experts[l] + e*expert_bytes (page-locked host memory) to
 * dev_experts[l] + e*expert_bytes (device), then resident[l*E+e] = nonzero
 * (when resident != NULL) and ready[l*E+e] = nonzero; per SPX_PLAN_EVICT,
 * ready[l*E+e] = 0 and resident[l*E+e] = 0.  The flags are host-to-device
 * copies from host_flags: 8 bytes of page-locked host memory holding
 * {1,0,0,0, 0,0,0,0} (the copy engines write them, so no SM is needed while
 * an expert launch that waits for them holds every SM).  ready/resident are device
 * arrays [L][E]; pass ready + l*E (and resident + l*E) to layer l's verify
 * call (spx_layer_args), whose expert launch waits for each routed expert's
 * flag.  For the FP16 packed experts of spx_f16_repack, expert_bytes =
 * spx_f16_packed_bytes(1, H, I) (expert e's units are contiguous).  Every
 * action is checked before anything is enqueued. */
SPX_API int spx_prefetch_issue(const int32_t *actions, int n_actions, const void *const *host_experts,
                               void *const *dev_experts, size_t expert_bytes, uint32_t *ready, uint8_t *resident,
                               const uint8_t *host_flags, int L, int E, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Gather tokens by expert (counting sort)  [P1 Key Contributions 4]         */
/* ------------------------------------------------------------------------ */
/* Flat slots s = t*k + j.  counts [E]: assignments per expert; offsets [E+1]:
 * exclusive prefix sum (offsets[E] = T*k); sorted_slots [T*k]: slots in
 * ascending expert, then ascending slot order ("sorted position" p indexes
 * this array); active [E]: experts with count > 0 in ascending order, the
 * rest -1; n_active [1]: how many.  Bit-exact and deterministic. */
SPX_API int spx_gather_by_expert(const int32_t *topk_ids, int T, int k, int E,
                         int32_t *counts, int32_t *offsets, int32_t *sorted_slots,
                         int32_t *active, int32_t *n_active, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert weight formats                                                      */
/* ------------------------------------------------------------------------ */
/* Canonical inputs (what a checkpoint holds):
 *  INT4 draft experts [P2 What shipped: GPTQ INT4, group 128], zero point 8,
 *   no act-order: qweight int32 [E][K/8][N], code of row kk at bits
 *   4*(kk%8)..+3 of word (kk/8, n); scales fp16 [E][K/128][N];
 *   W[kk][n] = (code - 8) * scale[kk/128][n].  gate/up: K = H, N = I;
 *   down: K = I, N = H.
 *  FP16 experts (verify, shared): PyTorch [out][in]: gate/up [E][I][H],
 *   down [E][H][I].
 *
 * Packed (what the expert kernels stream).  The repack calls below rewrite a
 * canonical tensor set once, at load time, into "units": one unit = one
 * expert's I-slice of S intermediate columns (gate rows, up rows and the
 * matching down columns), stored contiguously so that one unit is a few large
 * bulk copies, and laid out in the register-fragment order of the
 * m16n8k16 tensor-core instruction, so each lane reads its operands with
 * sequential 16-byte shared-memory loads.  The INT4 codes are re-packed two
 * fp16 lanes at a time for the magic-exponent dequantisation.  The byte order
 * inside a unit is private to the library; only the sizes below are public.
 *   INT4: S = 16 or 32 (slice_cols); unit bytes = 49*H*S/32; then the down
 *         scales, copied unchanged ([E][I/128][H] fp16); then the down
 *         weights once more in output-block order with their scales inline
 *         (read by the draft launch, whose reduction over I stays in a block).
 *   FP16: S = 16; unit bytes = 6*H*S.
 */
typedef struct {
    const void *packed; /* spx_w4_packed_bytes() bytes, from spx_w4_repack() */
    int E, H, I;        /* experts, hidden size, expert intermediate size */
    int slice_cols;     /* S: 16 or 32 */
    /* Per-group zero points (asymmetric INT4, the AWQ form: W = (code - zero)
     * * scale) [P1 Main Findings: drafts quantised by GPTQ, AWQ and GGUF]:
     * spx_w4_zeros_bytes() bytes from spx_w4_zeros_repack(), or NULL for zero
     * point 8.  Served by the one-launch draft path (T <= 5) and by the
     * expert launch (more tokens, cache-aware calls; 32-column slices take at
     * most 24 tokens there, else SPX_ERR_UNSUPPORTED). */
    const void *zeros;
} spx_w4_experts;

typedef struct {
    const void *packed; /* spx_f16_packed_bytes() bytes, from spx_f16_repack() */
    int E, H, I;
    /* Optional (NULL = none): the same experts in the tile pack of the
     * tensor-memory launches (spx_f16_tc_repack; I % 64 == 0).  With it (and
     * the shared expert's, when there is one) a verify layer call can run on
     * those launches (tcgen05 products, operands by TMA tensor copies): calls
     * of 9 to 64 tokens by default, any call with
     * spx_layer_args.verify_launch = 2. */
    const void *tc_packed;
} spx_f16_experts;

/* GGUF draft experts [P1 Main Findings: GGUF drafts at Q2, Q4 and Q8].
 * Canonical input per matrix, uint8 on the device, PyTorch [out][in] order
 * (each row holds the `in` weights of one output):
 *   Q8_0: a row is in/32 blocks of 34 bytes, a binary16 scale d
 *     (little-endian) then 32 signed 8-bit codes; weight j = d * code[j].
 *   Q2_K: a row is in/256 super-blocks of 84 bytes: 16 bytes, one per
 *     sub-block of 16 weights (low nibble scale sc, high nibble min m); 64
 *     bytes of 2-bit codes, weight w's code at bits 2*((w % 128) / 32) of byte
 *     32*(w / 128) + w % 32; binary16 d; binary16 dmin (little-endian);
 *     weight = d * sc * q - dmin * m.  Needs in % 256 == 0.
 *   Q4_K: a row is in/256 super-blocks of 144 bytes: binary16 d, binary16
 *     dmin, 12 bytes of 6-bit scales and mins of the 8 sub-blocks of 32
 *     weights (s < 4: scale = b[s] & 63, min = b[s+4] & 63; s >= 4: scale =
 *     (b[s+4] & 15) | (b[s-4] >> 6) << 4, min = (b[s+4] >> 4) | (b[s] >> 6)
 *     << 4), then 128 bytes of 4-bit codes, weight w in byte 32*(w / 64) +
 *     w % 32, low nibble when w % 64 < 32, else high nibble; weight =
 *     d * scale * q - dmin * min.  Needs in % 256 == 0.
 * gate and up are in gate_up_type ([E][I][H/32][34], [E][I][H/256][84] or
 * [E][I][H/256][144]);
 * down is Q8_0 ([E][H][I/32][34]): the down rows of the 1408-wide shapes are
 * not a multiple of 256.  Repacked (spx_gguf_repack) into the draft launch's
 * streaming order, 16 columns per slice, followed by the Q8_0 down weights in
 * the expert launch's unit order.  Served by the one-launch draft path (T <=
 * 5) and by the expert launch (more tokens, cache-aware calls). */
enum { SPX_GGUF_Q8_0 = 0, SPX_GGUF_Q2_K = 1, SPX_GGUF_Q4_K = 2 };
typedef struct {
    const void *packed; /* spx_gguf_packed_bytes() bytes, from spx_gguf_repack() */
    int E, H, I;
    int gate_up_type;   /* SPX_GGUF_Q8_0, SPX_GGUF_Q2_K or SPX_GGUF_Q4_K */
} spx_gguf_experts;

/* Shared expert(s): one FP16 MLP of intermediate size I_s (several shared
 * experts concatenated along I are one MLP, as the intermediate sum splits).
 * If w_sgate != NULL (fp16 [H]) its output is scaled per token by
 * gamma_t = 1 / (1 + exp(-x_t . w_sgate)).  [P1 Key Contributions 2] */
typedef struct {
    const void *packed;      /* spx_shared_packed_bytes(H, I_s) bytes, from spx_shared_repack() */
    const uint16_t *w_sgate; /* nullable; 16-byte aligned */
    int H, I_s;
    /* Optional (NULL = none): the shared expert in the tile pack of the
     * tensor-memory launches (spx_shared_tc_repack; I_s % 64 == 0); needed,
     * with the routed experts' one, by those launches. */
    const void *tc_packed;
} spx_shared;

SPX_API size_t spx_w4_packed_bytes(int E, int H, int I, int slice_cols);
SPX_API size_t spx_f16_packed_bytes(int E, int H, int I);
/* H, I multiples of 128 (Q2_K, Q4_K: H of 256); else 0 */
SPX_API size_t spx_gguf_packed_bytes(int E, int H, int I, int gate_up_type);
/* Shared expert pack: the FP16 units of one expert followed by its down
 * weights once more in output-block order (read by the draft launch). */
SPX_API size_t spx_shared_packed_bytes(int H, int I_s);

/* Repack canonical GPTQ tensors (device memory, layouts above) into `packed`
 * (device, spx_w4_packed_bytes() bytes, 16-byte aligned).  Deterministic. */
SPX_API int spx_w4_repack(const int32_t *qw_gate, const uint16_t *s_gate,
                  const int32_t *qw_up, const uint16_t *s_up,
                  const int32_t *qw_down, const uint16_t *s_down,
                  int E, int H, int I, int slice_cols, void *packed, spx_stream_t stream);

/* Zero points of asymmetric INT4 experts: canonical qzeros [E][K/128][N/8]
 * int32 per matrix (gate/up: K = H, N = I; down: K = I, N = H), the zero
 * point of column n in group g at bits 4*(n%8)..+3 of word (g, n/8), low
 * nibble first.  Repacked (device, 16-byte aligned) into the order the draft
 * launch streams them, next to the packed scales' order; deterministic. */
SPX_API size_t spx_w4_zeros_bytes(int E, int H, int I, int slice_cols);
SPX_API int spx_w4_zeros_repack(const int32_t *qz_gate, const int32_t *qz_up, const int32_t *qz_down,
                                int E, int H, int I, int slice_cols, void *zeros, spx_stream_t stream);

/* Repack canonical GGUF experts (layouts above spx_gguf_experts) into
 * `packed` (device, 16-byte aligned, spx_gguf_packed_bytes() bytes);
 * deterministic. */
SPX_API int spx_gguf_repack(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down, int E, int H, int I,
                            int gate_up_type, void *packed, spx_stream_t stream);

/* Repack one canonical FP16 shared expert ([I_s][H], [I_s][H], [H][I_s]) into
 * `packed` (device, spx_shared_packed_bytes() bytes, 16-byte aligned). */
SPX_API int spx_shared_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                              int H, int I_s, void *packed, spx_stream_t stream);

/* Repack canonical FP16 [out][in] tensors into `packed` (spx_f16_packed_bytes). */
SPX_API int spx_f16_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                   int E, int H, int I, void *packed, spx_stream_t stream);

/* Tile pack of the tensor-memory verify launches [P1 Key Contributions 4:
 * expert-wise verification as one dense product per expert].  Per expert:
 * the gate/up tiles (unit u = 64 columns of I, k-chunk kc = 64 rows of H, in
 * that order), then the down tiles (128-row block hb of H, k-chunk kc = 64
 * columns of I); a tile is 128 rows x 64 fp16 (16 KB), row-major.  Gate/up
 * tile row 32q + i (q < 4) holds gate column 64u + 16q + i for i < 16 and up
 * column 64u + 16q + i - 16 for i >= 16.  Bytes = E * 3 * I * H * 2 (the
 * canonical matrices' size); 0 if H % 128 or I % 64. */
SPX_API size_t spx_f16_tc_packed_bytes(int E, int H, int I);
/* Canonical [E][I][H], [E][I][H], [E][H][I] fp16 (16-byte aligned) into
 * `tc_packed` (device, spx_f16_tc_packed_bytes() bytes, 16-byte aligned). */
SPX_API int spx_f16_tc_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                              int E, int H, int I, void *tc_packed, spx_stream_t stream);
/* The shared expert ([I_s][H], [I_s][H], [H][I_s]): the pack of one expert,
 * spx_f16_tc_packed_bytes(1, H, I_s) bytes. */
SPX_API int spx_shared_tc_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                                 int H, int I_s, void *tc_packed, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Workspace                                                                  */
/* ------------------------------------------------------------------------ */
/* Bytes of workspace for calls with up to T tokens of hidden size H, routed
 * experts of intermediate size I (E of them, top-k) and a shared expert of
 * intermediate size I_s (0 = none); 0 if the shape is outside the limits. */
SPX_API size_t spx_workspace_size(int T, int H, int I, int E, int k, int I_s);
/* Bytes of workspace for a verify layer call forced onto the tensor-memory
 * launches (spx_layer_args.verify_launch = 2) with T tokens; equal to
 * spx_workspace_size() from T = 9 on.  0 if the shape cannot take them
 * (I or I_s not a multiple of 64, or outside the limits). */
SPX_API size_t spx_workspace_size_tc(int T, int H, int I, int E, int k, int I_s);
/* Zero a workspace; required once before first use (kernels leave it zeroed
 * again on exit) and after any call whose status word reported an error. */
SPX_API int spx_workspace_init(void *ws, size_t ws_bytes, spx_stream_t stream);
/* Asynchronously copy the workspace status word (SPX_OK or SPX_ERR_TIMEOUT)
 * into *host_status (page-locked host memory or device memory). */
SPX_API int spx_workspace_status(const void *ws, int32_t *host_status, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert MLPs   [P1 Key Contributions 4; P2 What shipped]                    */
/* ------------------------------------------------------------------------ */
/* For every assignment (t, e = topk_ids[t][j]):
 *   y = W_down_e( silu(W_gate_e x_t) * (W_up_e x_t) ),  silu(z) = z/(1+e^-z),
 * accumulated in fp32; the intermediate is rounded to fp16 before the down
 * projection (W4A16: dequantised INT4 weights times fp16 activations).
 * offsets/sorted_slots/active/n_active come from spx_gather_by_expert.
 * Output: y_sorted fp32 [T*k][H], row p = the assignment sorted_slots[p]
 * (zeroed by the call, then accumulated).
 *
 * draft: one fused launch over all active experts' INT4 units.
 * verify: the same launch shape over FP16 experts; each active expert's
 *   weights are read once for all of its n_e tokens (expert-wise reordering:
 *   tokens of one expert form the columns of one tensor-core product). */
SPX_API int spx_moe_draft_w4a16(const uint16_t *x, int T, const spx_w4_experts *w, int k,
                        const int32_t *offsets, const int32_t *sorted_slots,
                        const int32_t *active, const int32_t *n_active,
                        float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream);

/* The draft unit call with GGUF experts (the draft launch up to 5 tokens,
 * the expert launch above); arguments and output as spx_moe_draft_w4a16. */
SPX_API int spx_moe_draft_gguf(const uint16_t *x, int T, const spx_gguf_experts *w, int k,
                        const int32_t *offsets, const int32_t *sorted_slots,
                        const int32_t *active, const int32_t *n_active,
                        float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream);

SPX_API int spx_moe_verify_fp16(const uint16_t *x, int T, const spx_f16_experts *w, int k,
                        const int32_t *offsets, const int32_t *sorted_slots,
                        const int32_t *active, const int32_t *n_active,
                        float *y_sorted, void *ws, size_t ws_bytes, spx_stream_t stream);

/* Weighted scatter-combine plus shared expert:
 *   out[t] = fp16( sum_j topk_w[t][j] * y_sorted[pos(t,j)] + gamma_t * sh_t )
 * where pos(t,j) is the sorted position of slot t*k+j and sh_t the shared
 * expert MLP of x_t (omitted when shared == NULL).  out: fp16 [T][H]. */
SPX_API int spx_combine(const float *y_sorted, const int32_t *sorted_slots, const float *topk_w,
                const uint16_t *x, const spx_shared *shared, int T, int H, int k,
                uint16_t *out, void *ws, size_t ws_bytes, spx_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Composite layer: route, top-k, counters, gather, experts, shared, combine  */
/* ------------------------------------------------------------------------ */
typedef struct {
    int mode;                  /* 0 = draft (INT4 routed experts), 1 = verify (FP16) */
    int T, H, E, k, renorm;
    const uint16_t *x;         /* [T][H] fp16 */
    const uint16_t *w_router;  /* [E][H] fp16, or NULL: logits are given */
    float *logits;             /* [T][E]: output if w_router, else input */
    const spx_w4_experts *w4;  /* mode 0 */
    const spx_f16_experts *f16;/* mode 1 */
    const spx_shared *shared;  /* NULL = no shared expert */
    uint32_t *elb;             /* [L][E] counters to update, or NULL */
    int L, layer;
    /* routing outputs (caller-owned, same meaning as the unit calls) */
    int32_t *topk_ids;         /* [T][k] */
    float *topk_w;             /* [T][k] */
    int32_t *counts;           /* [E] */
    int32_t *offsets;          /* [E+1] */
    int32_t *sorted_slots;     /* [T*k] */
    int32_t *active;           /* [E] */
    int32_t *n_active;         /* [1] */
    uint16_t *out;             /* [T][H] fp16 */
    void *ws;
    size_t ws_bytes;
    /* Instrumentation, both nullable: cudaEvent_t handles recorded on the
     * stream immediately before and after the expert launch (recording between
     * the two launches removes their programmatic overlap). */
    void *ev_experts_begin;
    void *ev_experts_end;
    /* Cache-aware expert execution [P1 Key Contributions 3-4: experts the
     * lookahead saw are cache hits and run first; misses wait for their
     * weights].  Both nullable; when either is set the layer runs as a routing
     * launch plus the expert launch (also for draft calls of T <= 5).
     *   resident [E] uint8: nonzero = expert e's weights are resident; the
     *     routed experts are queued resident first, then the others, each in
     *     ascending expert order.  Only the order changes, not the result.
     *   ready [E] uint32: before it streams expert e's weights the expert
     *     launch waits until ready[e] is nonzero (the caller sets it once the
     *     weights have landed, e.g. by a copy on another stream); a wait longer
     *     than the bound below stops the launch with SPX_ERR_TIMEOUT in the
     *     workspace status word (the output is then undefined). */
    const uint8_t *resident;
    const uint32_t *ready;
    /* Bound of every device-side wait of the call in ns; 0 = 2 s. */
    uint64_t wait_budget_ns;
    /* mode 0 with GGUF draft experts instead of INT4 (w4 must then be NULL). */
    const spx_gguf_experts *gguf;
    /* mode 1: which launches run the experts.  0 = automatic (the
     * tensor-memory launches for 9 to 64 tokens when the tile packs are given
     * and no cache-aware option is set, else the expert launch); 1 = the
     * expert launch; 2 = the tensor-memory launches (tile packs required, no
     * cache-aware options, ws_bytes at least spx_workspace_size_tc(); else
     * SPX_ERR_UNSUPPORTED / SPX_ERR_WORKSPACE). */
    int verify_launch;
} spx_layer_args;

/* One layer.  Draft calls with T <= 5 (and no cache-aware options) are one
 * launch that routes its tokens in every block (after a router-product launch
 * when w_router is given); other calls are a routing launch (router product,
 * softmax, top-k, counters, counting sort, token tables) and then either one
 * persistent expert launch that streams the shared expert first, then every
 * active expert's units, and writes out[] from its last blocks, or (verify
 * calls of 9+ tokens with the tile packs, see verify_launch) the
 * tensor-memory launches: a gather of each expert's token rows, one
 * persistent tcgen05 launch for every expert's gate/up and then down products
 * [P1 Key Contributions 4], and an output launch.  Every launch of the call
 * may begin while the one before it on the stream finishes (programmatic
 * dependent launch): it reads nothing that launch writes before it has
 * completed. */
SPX_API int spx_moe_layer(const spx_layer_args *args, spx_stream_t stream);

/* The same layer for callers that cannot allocate device memory (code running
 * inside an allocator or pool callback, runtimes that forbid device allocation
 * after start-up, hosts that must not wait on the allocator).  The paper has no
 * counterpart; it is a deployment convenience of this library.
 * args->ws and args->ws_bytes are ignored: the scratch is a fixed 1 MiB array
 * inside the library image, present on every GPU that loads the library until
 * the process exits.  Shapes whose workspace exceeds 1 MiB are rejected with
 * SPX_ERR_WORKSPACE (the DeepSeek-V2-Lite-shaped layer fits at T = 1 and T =
 * 17); a verify call left to the automatic choice whose tensor-memory
 * launches' scratch (spx_workspace_size_tc) would not fit takes the expert
 * launch, whose workspace is the smaller one.  The call allocates nothing, provided
 * spx_noalloc_init() has run on the current device first; on a device where it
 * has not, the call returns SPX_ERR_WORKSPACE and enqueues nothing.  Arguments
 * are checked before anything is enqueued; then the call clears the part of
 * the array that must start at zero.  Every call shares the one array, which
 * keeps the last call's contents, so calls that can overlap on the GPU (two
 * streams, two host threads) race on it.  A bounded device-side wait that
 * gives up is reported in the array's status word: read it with
 * spx_noalloc_status() after the call, before the next one. */
SPX_API int spx_moe_layer_noalloc(const spx_layer_args *args, spx_stream_t stream);
/* Set-up of spx_moe_layer_noalloc for the current device, once per device at
 * start-up, before any stream capture: loads every kernel the layer call can
 * launch and the fixed scratch array onto the device (this allocates device
 * memory for the library's code and the array, which is why it is a call of
 * its own) and looks up the array's address.  Later calls on the device
 * return SPX_OK at once.  After cudaDeviceReset, call it again.  No
 * counterpart in the paper. */
SPX_API int spx_noalloc_init(void);
/* Asynchronously copy the fixed scratch array's status word (SPX_OK or
 * SPX_ERR_TIMEOUT) of the current device into *status (page-locked host
 * memory or device memory), ordered on `stream` after the layer calls before
 * it; SPX_ERR_WORKSPACE if spx_noalloc_init has not run on the device.  No
 * counterpart in the paper. */
SPX_API int spx_noalloc_status(int32_t *status, spx_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPX_H */
