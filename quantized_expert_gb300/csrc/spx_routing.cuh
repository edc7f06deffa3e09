// spx_routing.cuh -- per-token softmax + top-k, shared by the routing launch
// and by the draft launch, which routes its few tokens inside every block.
//
// Method (ai.info summary of the Specter paper, Key Contributions 2-4; the
// draft shares the target's router): the k experts with the largest logits,
// ties to the lower expert index; softmax over all E experts; the selected
// weights, renormalised over the k selected when the model does so.
#pragma once

#include "spx_internal.cuh"

#include <math.h>

namespace spx {

#if defined(__CUDACC__)
// Order key of a logit: unsigned compare of keys = float compare of values
// (-0 is taken as +0); 0 marks an expert already taken or absent.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Warp-collective selection for one token.  lg(e) returns logit e (fp32, the
// precision every decision is taken in); E <= 256, k <= E.  The experts are
// taken in the order (value descending, index ascending): k rounds, each a
// warp-wide maximum of the order keys, ties to the lowest expert index.
// p = expf(v - max) / sum over all E of expf(v - max) (each lane sums its
// experts e = lane + 32 j in j order, then a fixed xor-shuffle tree);
// weight = p, or p / (sum of the k selected p, in rank order) when renorm.
// The lane owning the rank-r expert writes ids[r] and w[r]; sv (E floats of
// shared scratch) is not used.
template <int NPER, class Logit>
__device__ __forceinline__ void select_token_n(Logit lg, int E, int k, int renorm, int lane, int32_t *ids, float *w,
                                               float *sv) {
    (void)sv;
    float v[NPER];
    uint32_t key[NPER];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? lg(e) : -INFINITY;
        key[j] = e < E ? logit_key(v[j]) : 0u;
        if (e < E) m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (lane + 32 * j < E) z += expf(v[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    for (int r = 0; r < k; ++r) {
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < NPER; ++j)
            if (key[j] > bk) {  // strict: the lowest j among equal keys
                bk = key[j];
                bj = j;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t win = __reduce_min_sync(0xffffffffu, (bk == mk && mk != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu);
        if ((int)(win & 31u) == lane && win != 0xffffffffu) {
#pragma unroll
            for (int j = 0; j < NPER; ++j)
                if (j == (int)(win >> 5)) {
                    ids[r] = (int32_t)win;
                    w[r] = expf(v[j] - m) / z;
                    key[j] = 0u;
                }
        }
    }
    __syncwarp();
    if (lane == 0 && renorm) {
        float psel = 0.f;
        for (int r = 0; r < k; ++r) psel += w[r];
        for (int r = 0; r < k; ++r) w[r] = w[r] / psel;
    }
    __syncwarp();
}

// Selection for one token by several warps of a block (E <= 64): sv holds
// the token's E logits in shared memory.  Each calling warp computes the
// maximum and the softmax sum exactly as select_token_n does, and ranks eight
// experts e = 8 w + lane/4 (four lanes per expert, each counting a quarter
// of the others; rank = experts before e in the order value descending,
// index ascending); the lane holding a rank-r expert (r < k) writes ids[r]
// and its softmax weight w[r] (renormalisation is left to the caller, once
// every warp is done).  Warps w >= E/8 have nothing to rank and may skip it.
__device__ __forceinline__ void select_rank_warp(const float *sv, int E, int k, int w, int lane, int32_t *ids,
                                                 float *wout) {
    float v[2];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? sv[e] : -INFINITY;
        if (e < E) m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if (lane + 32 * j < E) z += expf(v[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const int e = 8 * w + (lane >> 2), q = lane & 3;
    const float ve = e < E ? sv[e] : 0.f;
    int rank = 0;
    if (e < E)
        for (int e2 = q; e2 < E; e2 += 4) {
            const float u = sv[e2];
            rank += (u > ve || (u == ve && e2 < e)) ? 1 : 0;
        }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (e < E && q == 0 && rank < k) {
        ids[rank] = e;
        wout[rank] = expf(ve - m) / z;
    }
}

template <class Logit>
__device__ __forceinline__ void select_token(Logit lg, int E, int k, int renorm, int lane, int32_t *ids, float *w,
                                             float *sv) {
    switch ((E + 31) >> 5) {  // experts per lane, a compile-time count below
        case 1: select_token_n<1>(lg, E, k, renorm, lane, ids, w, sv); break;
        case 2: select_token_n<2>(lg, E, k, renorm, lane, ids, w, sv); break;
        case 3: select_token_n<3>(lg, E, k, renorm, lane, ids, w, sv); break;
        case 4: select_token_n<4>(lg, E, k, renorm, lane, ids, w, sv); break;
        case 5:
        case 6: select_token_n<6>(lg, E, k, renorm, lane, ids, w, sv); break;
        default: select_token_n<8>(lg, E, k, renorm, lane, ids, w, sv); break;
    }
}

// The same selection for logits in global memory (one token's row), kept out
// of line with one instance (up to 8 experts per lane): a kernel that selects
// once per launch keeps its hot loops close together in the instruction
// cache instead of carrying an unrolled copy per expert count.
static __device__ __noinline__ void select_token_global(const float *logits, int E, int k, int renorm, int lane,
                                                 int32_t *ids, float *w) {
    select_token_n<8>([&](int e) { return __ldcg(logits + e); }, E, k, renorm, lane, ids, w, nullptr);
}
#endif  // __CUDACC__

}  // namespace spx
