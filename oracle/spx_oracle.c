/*
 * spx_oracle.c -- CPU oracle for the Specter per-layer MoE expert path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
 * restatement of what the path computes, used by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg.  The CUDA library never
 * links, includes or calls it, and it shares no code with the library.
 *
 * Arithmetic is IEEE binary64 throughout (the pages fix no precision for a
 * reference); inputs arrive as fp16 bit patterns, int32 GPTQ words and fp32
 * logits.  Where a floating-point value decides an integer (the top-k
 * selection), the decision is taken on the fp32 value, as the kernels do.
 *
 * Sources, cited by page title and section:
 *  [S1] ai.info, "Specter: Fast MoE Inference via Quantization-Enabled
 *       Multi-Step Speculative Offloading" (AI summary): Key Contributions
 *       items 1-4 and "Methodology in Plain English" -- INT4 copy of the
 *       target's experts as draft, FP16 gates and shared experts, GPU-side
 *       per-layer expert-activation counters (the Expert Lookahead Buffer),
 *       tokens gathered by expert and computed in one fused draft launch,
 *       expert-wise packing of verification tokens ("mathematically
 *       identical").
 *  [S2] richland.au, "Specter previews expert routing with an INT4 copy of
 *       the model itself", section "What shipped" -- GPTQ INT4, group size
 *       128, routers and shared experts reuse the target's FP16 tensors,
 *       W4A16 kernels that dequantise INT4 tiles and compute in FP16.
 *  Readings where the pages are silent (top-k key and tie order, renorm,
 *  GPTQ nibble order and zero point, SwiGLU form, combine) are listed
 *  beside each function and in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary64                                       */
/* ------------------------------------------------------------------ */

/* Decode a binary16 bit pattern: sign, 5-bit biased exponent (bias 15),
 * 10-bit fraction; exponent 0 = subnormal (fraction * 2^-24), 31 = inf/NaN. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(fr | 0x400), ex - 25);
    return sign ? -v : v;
}

/* Encode to binary16 with round-to-nearest, ties-to-even. */
uint16_t orc_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds to even = inf */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal: quantum 2^-24; rint() is ties-to-even in the default mode.
         * A result of 1024 is the bit pattern of the smallest normal. */
        double m = rint(ldexp(a, 24));
        return sign | (uint16_t)m;
    }
    int e2;
    frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;          /* a in [2^E, 2^(E+1)) */
    double m = rint(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (m >= 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E + 15 >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024));
}

void orc_halves_to_doubles(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_half_to_double(in[i]);
}

void orc_doubles_to_halves(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_double_to_half(in[i]);
}

/* decode table, filled from orc_half_to_double on first use */
static double g_half_tab[65536];
static int g_half_tab_ready = 0;

static const double *half_tab(void)
{
    if (!g_half_tab_ready) {
        for (int i = 0; i < 65536; ++i)
            g_half_tab[i] = orc_half_to_double((uint16_t)i);
        g_half_tab_ready = 1;
    }
    return g_half_tab;
}

/* ------------------------------------------------------------------ */
/* Router: logits, softmax, top-k, weights  [S1 Key Contributions 2;    */
/* S2 What shipped: routers reuse the target's FP16 tensors]           */
/* ------------------------------------------------------------------ */

/* logits[t][e] = sum_h x[t][h] * wr[e][h], h ascending. */
void orc_router_logits(const uint16_t *x, const uint16_t *wr, int T, int H, int E, double *logits)
{
    const double *tab = half_tab();
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += tab[x[(int64_t)t * H + h]] * tab[wr[(int64_t)e * H + h]];
            logits[(int64_t)t * E + e] = acc;
        }
}

/* Reading: the k experts with the largest logits (logits rounded to fp32,
 * the precision the kernels decide in), ties to the lower expert index,
 * listed in descending order; softmax over all E experts in fp64;
 * weight = p[id], or p[id] / sum of the selected p when renorm != 0.
 * probs (nullable) receives the full softmax [T][E]. */
void orc_route_topk(const double *logits, int T, int E, int k, int renorm,
                    int32_t *ids, double *w, double *probs)
{
    float *lf = (float *)malloc(sizeof(float) * (size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e)
            lf[e] = (float)logits[(int64_t)t * E + e];
        /* softmax */
        double m = -INFINITY;
        for (int e = 0; e < E; ++e)
            if ((double)lf[e] > m)
                m = (double)lf[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = exp((double)lf[e] - m);
            z += p[e];
        }
        for (int e = 0; e < E; ++e)
            p[e] /= z;
        if (probs)
            for (int e = 0; e < E; ++e)
                probs[(int64_t)t * E + e] = p[e];
        /* stable insertion sort of expert indices by descending fp32 logit;
         * equal logits keep ascending index order (lower index first) */
        for (int e = 0; e < E; ++e) {
            int j = e;
            while (j > 0 && lf[order[j - 1]] < lf[e]) {
                order[j] = order[j - 1];
                --j;
            }
            order[j] = e;
        }
        double sel = 0.0;
        for (int j = 0; j < k; ++j)
            sel += p[order[j]];
        for (int j = 0; j < k; ++j) {
            ids[(int64_t)t * k + j] = order[j];
            w[(int64_t)t * k + j] = renorm ? p[order[j]] / sel : p[order[j]];
        }
    }
    free(lf);
    free(p);
    free(order);
}

/* ------------------------------------------------------------------ */
/* Expert Lookahead Buffer: layer-indexed activation counters           */
/* [S1 Key Contributions 3; Methodology: counters tally how often each  */
/* expert in each layer is selected as draft tokens are generated]      */
/* ------------------------------------------------------------------ */

/* elb is [L][E]; one increment per (token, slot) selection. */
void orc_elb_accumulate(uint32_t *elb, int E, int layer, const int32_t *ids, int T, int k)
{
    for (int s = 0; s < T * k; ++s)
        elb[(int64_t)layer * E + ids[s]] += 1u;
}

/* ------------------------------------------------------------------ */
/* Gather tokens by expert [S1 Key Contributions 4: the fused draft     */
/* kernel gathers tokens by expert; verification packs tokens routed    */
/* to the same expert together]                                         */
/* ------------------------------------------------------------------ */

/* Counting sort of the flat slots s = t*k + j by expert id: counts[e];
 * offsets = exclusive prefix sum (E+1 entries); sorted_slots lists slots
 * in ascending expert, then ascending slot order; active lists the experts
 * with count > 0 in ascending order, n_active of them. */
void orc_gather_by_expert(const int32_t *ids, int T, int k, int E, int32_t *counts,
                          int32_t *offsets, int32_t *sorted_slots, int32_t *active,
                          int32_t *n_active)
{
    int n = T * k;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int s = 0; s < n; ++s)
        counts[ids[s]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e)
        fill[e] = offsets[e];
    for (int s = 0; s < n; ++s)
        sorted_slots[fill[ids[s]]++] = s;
    free(fill);
    int a = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0)
            active[a++] = e;
    for (int e = a; e < E; ++e)
        active[e] = -1;
    *n_active = a;
}

/* ------------------------------------------------------------------ */
/* GPTQ INT4, group 128, zero point 8  [S2 What shipped]                */
/* ------------------------------------------------------------------ */

/* Reading: qweight is [K/8][N] int32, code of row kk at bits 4*(kk%8)..+3
 * of word (kk/8, n), low nibble first; scales [K/128][N] fp16; no act-order
 * permutation; W[kk][n] = (code - 8) * scale[kk/128][n]. */
static inline double w4_at(const int32_t *q, const uint16_t *s, const double *tab, int N, int kk, int n)
{
    uint32_t word = (uint32_t)q[(int64_t)(kk / 8) * N + n];
    int code = (int)((word >> (4 * (kk % 8))) & 15u);
    return (double)(code - 8) * tab[s[(int64_t)(kk / 128) * N + n]];
}

/* Asymmetric INT4 (per-group zero points, the AWQ form of the same codes;
 * [S1 Main Findings: drafts quantised by GPTQ, AWQ and GGUF]).  Reading: qzeros is
 * [K/128][N/8] int32, the zero point of column n in group g at bits
 * 4*(n%8)..+3 of word (g, n/8), low nibble first;
 * W[kk][n] = (code - zero) * scale[kk/128][n].  qz == NULL: zero point 8. */
static inline double w4z_at(const int32_t *q, const uint16_t *s, const int32_t *qz, const double *tab, int N,
                            int kk, int n)
{
    if (!qz)
        return w4_at(q, s, tab, N, kk, n);
    uint32_t word = (uint32_t)q[(int64_t)(kk / 8) * N + n];
    int code = (int)((word >> (4 * (kk % 8))) & 15u);
    uint32_t zword = (uint32_t)qz[(int64_t)(kk / 128) * (N / 8) + n / 8];
    int zero = (int)((zword >> (4 * (n % 8))) & 15u);
    return (double)(code - zero) * tab[s[(int64_t)(kk / 128) * N + n]];
}

/* out[kk][n] = W[kk][n] for the whole K x N matrix (qz nullable). */
void orc_w4z_dequant(const int32_t *q, const uint16_t *s, const int32_t *qz, int K, int N, double *out)
{
    const double *tab = half_tab();
    for (int kk = 0; kk < K; ++kk)
        for (int n = 0; n < N; ++n)
            out[(int64_t)kk * N + n] = w4z_at(q, s, qz, tab, N, kk, n);
}

void orc_w4_dequant(const int32_t *q, const uint16_t *s, int K, int N, double *out)
{
    orc_w4z_dequant(q, s, NULL, K, N, out);
}

/* ------------------------------------------------------------------ */
/* Expert MLP: y = W_down ( silu(W_gate x) * (W_up x) )                 */
/* Reading: SwiGLU, the MLP form of all three named models; silu(z) =   */
/* z / (1 + exp(-z)); the intermediate h is kept in fp64.              */
/* ------------------------------------------------------------------ */

static inline double silu(double z) { return z / (1.0 + exp(-z)); }

/* INT4 expert (GPTQ layout, gate/up K=H N=I, down K=I N=H) on one token;
 * zg, zu, zd: per-group zero points (nullable: zero point 8). */
void orc_swiglu_w4z(const uint16_t *x, int H, int I,
                    const int32_t *qg, const uint16_t *sg, const int32_t *zg,
                    const int32_t *qu, const uint16_t *su, const int32_t *zu,
                    const int32_t *qd, const uint16_t *sd, const int32_t *zd,
                    double *y, double *h_out)
{
    const double *tab = half_tab();
    double *g = (double *)calloc((size_t)I, sizeof(double));
    double *u = (double *)calloc((size_t)I, sizeof(double));
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    /* g[i] = sum_kk W_g[kk][i] x[kk], kk ascending for every i */
    for (int kk = 0; kk < H; ++kk) {
        double xk = tab[x[kk]];
        for (int i = 0; i < I; ++i) {
            g[i] += w4z_at(qg, sg, zg, tab, I, kk, i) * xk;
            u[i] += w4z_at(qu, su, zu, tab, I, kk, i) * xk;
        }
    }
    for (int i = 0; i < I; ++i)
        h[i] = silu(g[i]) * u[i];
    for (int n = 0; n < H; ++n)
        y[n] = 0.0;
    for (int i = 0; i < I; ++i)
        for (int n = 0; n < H; ++n)
            y[n] += w4z_at(qd, sd, zd, tab, H, i, n) * h[i];
    if (h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(g);
    free(u);
    free(h);
}

void orc_swiglu_w4(const uint16_t *x, int H, int I,
                   const int32_t *qg, const uint16_t *sg,
                   const int32_t *qu, const uint16_t *su,
                   const int32_t *qd, const uint16_t *sd,
                   double *y, double *h_out)
{
    orc_swiglu_w4z(x, H, I, qg, sg, NULL, qu, su, NULL, qd, sd, NULL, y, h_out);
}

/* ------------------------------------------------------------------ */
/* GGUF Q8_0 experts [S1 Main Findings: GGUF drafts at Q2, Q4 and Q8].  */
/* Reading (the GGUF format definition; the pages name the format       */
/* only): a weight matrix in [out][in] order, each row of `in` values   */
/* cut into blocks of 32 consecutive values; a block is 34 bytes, the   */
/* binary16 scale d (little-endian) then 32 signed 8-bit codes, and     */
/* value j of the block is d * code[j].                                 */
/* ------------------------------------------------------------------ */

static inline double q8_at(const uint8_t *w, const double *tab, int K, int n, int kk)
{
    const uint8_t *blk = w + ((int64_t)n * (K / 32) + kk / 32) * 34;
    uint16_t d = (uint16_t)(blk[0] | (blk[1] << 8));
    int code = (int)(int8_t)blk[2 + kk % 32];
    return (double)code * tab[d];
}

/* out[n][kk] = W[n][kk] for an N x K matrix ([out][in]). */
void orc_q8_dequant(const uint8_t *w, int N, int K, double *out)
{
    const double *tab = half_tab();
    for (int n = 0; n < N; ++n)
        for (int kk = 0; kk < K; ++kk)
            out[(int64_t)n * K + kk] = q8_at(w, tab, K, n, kk);
}

/* GGUF Q2_K [S1 Main Findings: GGUF Q2 drafts].  Reading (the GGUF
 * format): a row is cut into super-blocks of 256 consecutive values, each
 * 84 bytes: 16 bytes of sub-block parameters, 64 bytes of 2-bit codes, then
 * the binary16 scale d and the binary16 min scale dmin (little-endian).
 * Sub-block b = 16 consecutive values; its byte holds the 4-bit scale sc
 * (low nibble) and the 4-bit min m (high nibble).  Value w of the
 * super-block has its code q (0..3) at bits 2*((w % 128) / 32) of code byte
 * 32*(w / 128) + w % 32, and equals d*sc*q - dmin*m.  Rows need a multiple
 * of 256 values. */
static inline double q2k_at(const uint8_t *w, const double *tab, int K, int n, int kk)
{
    const uint8_t *blk = w + ((int64_t)n * (K / 256) + kk / 256) * 84;
    int wi = kk % 256;
    int par = blk[wi / 16];
    int q = (blk[16 + 32 * (wi / 128) + wi % 32] >> (2 * ((wi % 128) / 32))) & 3;
    double d = tab[(uint16_t)(blk[80] | (blk[81] << 8))];
    double dmin = tab[(uint16_t)(blk[82] | (blk[83] << 8))];
    return d * (double)(par & 15) * (double)q - dmin * (double)(par >> 4);
}

/* GGUF Q4_K [S1 Main Findings: GGUF Q4 drafts].  Reading (the GGUF format):
 * super-blocks of 256 consecutive values in 144 bytes: binary16 d, binary16
 * dmin (little-endian), 12 bytes of 6-bit sub-block scales and mins, then
 * 128 bytes of 4-bit codes.  Sub-block s = 32 consecutive values (8 per
 * super-block).  For s < 4: scale = byte[s] & 63, min = byte[s+4] & 63; for
 * s >= 4: scale = (byte[s+4] & 15) | (byte[s-4] >> 6) << 4 and
 * min = (byte[s+4] >> 4) | (byte[s] >> 6) << 4 (bytes of the 12).  Value w:
 * chunk c = w / 64 uses code byte 32*c + w % 32, its low nibble for
 * w % 64 < 32 (sub-block 2c), its high nibble otherwise (sub-block 2c+1);
 * value = d*scale*q - dmin*min. */
static inline void q4k_scale_min(const uint8_t *sc12, int s, int *scale, int *mn)
{
    if (s < 4) {
        *scale = sc12[s] & 63;
        *mn = sc12[s + 4] & 63;
    } else {
        *scale = (sc12[s + 4] & 15) | ((sc12[s - 4] >> 6) << 4);
        *mn = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);
    }
}

static inline double q4k_at(const uint8_t *w, const double *tab, int K, int n, int kk)
{
    const uint8_t *blk = w + ((int64_t)n * (K / 256) + kk / 256) * 144;
    int wi = kk % 256;
    int scale, mn;
    q4k_scale_min(blk + 4, wi / 32, &scale, &mn);
    int byte = blk[16 + 32 * (wi / 64) + wi % 32];
    int q = (wi % 64) < 32 ? (byte & 15) : (byte >> 4);
    double d = tab[(uint16_t)(blk[0] | (blk[1] << 8))];
    double dmin = tab[(uint16_t)(blk[2] | (blk[3] << 8))];
    return d * (double)scale * (double)q - dmin * (double)mn;
}

/* out[n][kk] = W[n][kk] of a Q4_K matrix, N x K ([out][in]). */
void orc_q4k_dequant(const uint8_t *w, int N, int K, double *out)
{
    const double *tab = half_tab();
    for (int n = 0; n < N; ++n)
        for (int kk = 0; kk < K; ++kk)
            out[(int64_t)n * K + kk] = q4k_at(w, tab, K, n, kk);
}

/* Matrix value by format: ORC_Q8_0, ORC_Q2_K or ORC_Q4_K. */
enum { ORC_Q8_0 = 0, ORC_Q2_K = 1, ORC_Q4_K = 2 };
static inline double gguf_at(int type, const uint8_t *w, const double *tab, int K, int n, int kk)
{
    if (type == ORC_Q2_K)
        return q2k_at(w, tab, K, n, kk);
    if (type == ORC_Q4_K)
        return q4k_at(w, tab, K, n, kk);
    return q8_at(w, tab, K, n, kk);
}

/* out[n][kk] = W[n][kk] of a Q2_K matrix, N x K ([out][in]). */
void orc_q2k_dequant(const uint8_t *w, int N, int K, double *out)
{
    const double *tab = half_tab();
    for (int n = 0; n < N; ++n)
        for (int kk = 0; kk < K; ++kk)
            out[(int64_t)n * K + kk] = q2k_at(w, tab, K, n, kk);
}

/* GGUF expert on one token, each matrix in its own format (tg, tu, td):
 * wg, wu [I] rows of H values; wd [H] rows of I values. */
void orc_swiglu_gguf(const uint16_t *x, int H, int I, int tg, const uint8_t *wg, int tu, const uint8_t *wu, int td,
                     const uint8_t *wd, double *y, double *h_out)
{
    const double *tab = half_tab();
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int kk = 0; kk < H; ++kk) {
            double xk = tab[x[kk]];
            g += gguf_at(tg, wg, tab, H, i, kk) * xk;
            u += gguf_at(tu, wu, tab, H, i, kk) * xk;
        }
        h[i] = silu(g) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += gguf_at(td, wd, tab, I, n, i) * h[i];
        y[n] = acc;
    }
    if (h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(h);
}

/* Q8_0 expert on one token: wg, wu [I][H/32] blocks; wd [H][I/32] blocks. */
void orc_swiglu_q8(const uint16_t *x, int H, int I, const uint8_t *wg, const uint8_t *wu, const uint8_t *wd,
                   double *y, double *h_out)
{
    orc_swiglu_gguf(x, H, I, ORC_Q8_0, wg, ORC_Q8_0, wu, ORC_Q8_0, wd, y, h_out);
}

/* FP16 expert, PyTorch [out, in] layout: wg, wu [I][H]; wd [H][I]. */
void orc_swiglu_f16(const uint16_t *x, int H, int I,
                    const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                    double *y, double *h_out)
{
    const double *tab = half_tab();
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint16_t *rg = wg + (int64_t)i * H;
        const uint16_t *ru = wu + (int64_t)i * H;
        for (int kk = 0; kk < H; ++kk) {
            double xk = tab[x[kk]];
            g += tab[rg[kk]] * xk;
            u += tab[ru[kk]] * xk;
        }
        h[i] = silu(g) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        const uint16_t *rd = wd + (int64_t)n * I;
        for (int i = 0; i < I; ++i)
            acc += tab[rd[i]] * h[i];
        y[n] = acc;
    }
    if (h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(h);
}

/* Sigmoid gate of a gated shared expert: 1 / (1 + exp(-x . w)). */
double orc_shared_gate(const uint16_t *x, const uint16_t *wsg, int H)
{
    const double *tab = half_tab();
    double z = 0.0;
    for (int kk = 0; kk < H; ++kk)
        z += tab[x[kk]] * tab[wsg[kk]];
    return 1.0 / (1.0 + exp(-z));
}

/* ------------------------------------------------------------------ */
/* Weighted scatter-combine                                             */
/* Reading: out[t] = sum_j w[t][j] * y[t*k+j] + gamma[t] * sh[t], summed */
/* in ascending j, then rounded once to fp16.                           */
/* ------------------------------------------------------------------ */

void orc_combine(int T, int H, int k, const double *w, const double *y_slot,
                 const double *gamma, const double *sh, double *out, uint16_t *out_half)
{
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += w[(int64_t)t * k + j] * y_slot[((int64_t)t * k + j) * H + n];
            if (sh)
                acc += (gamma ? gamma[t] : 1.0) * sh[(int64_t)t * H + n];
            out[(int64_t)t * H + n] = acc;
            if (out_half)
                out_half[(int64_t)t * H + n] = orc_double_to_half(acc);
        }
}
