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
// Warp-collective selection for one token.  lg(e) returns logit e (fp32, the
// precision every decision is taken in); E <= 256, k <= E.  An expert's rank
// is the number of experts before it in the order (value descending, index
// ascending); the k experts of rank < k are the selection, listed by rank.
// p = expf(v - max) / sum over all E of expf(v - max) (each lane sums its
// experts e = lane + 32 j in j order, then a fixed xor-shuffle tree);
// weight = p, or p / (sum of the k selected p, in rank order) when renorm.
// sv is E floats of scratch in shared memory.  Lane 0 publishes nothing
// itself: the lanes owning selected experts write ids[rank] and w[rank].
template <int NPER, class Logit>
__device__ __forceinline__ void select_token_n(Logit lg, int E, int k, int renorm, int lane, int32_t *ids, float *w,
                                               float *sv) {
    float v[NPER];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? lg(e) : -INFINITY;
        if (e < E) {
            sv[e] = v[j];
            m = fmaxf(m, v[j]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (lane + 32 * j < E) z += expf(v[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    __syncwarp();
    int rank[NPER];
#pragma unroll
    for (int j = 0; j < NPER; ++j) rank[j] = 0;
#pragma unroll 4
    for (int e2 = 0; e2 < E; ++e2) {
        const float u = sv[e2];
#pragma unroll
        for (int j = 0; j < NPER; ++j) rank[j] += (u > v[j] || (u == v[j] && e2 < lane + 32 * j)) ? 1 : 0;
    }
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        if (e < E && rank[j] < k) {
            ids[rank[j]] = e;
            w[rank[j]] = expf(v[j] - m) / z;
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
#endif  // __CUDACC__

}  // namespace spx
