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

// Inverse of logit_key for a nonzero key (gives +0 for a -0 logit, which
// has the same softmax term).
__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Warp-collective selection for one token.  lg(e) returns logit e (fp32, the
// precision every decision is taken in); E <= 32 NPER, k <= E.  The experts
// are taken in the order (value descending, index ascending): k rounds, each
// a warp-wide maximum of the order keys; the lane holding it (expert
// e = lane + 32 j, its lowest such j) takes the round, and when several lanes
// hold it, the one with the lowest expert index does.  The round's winner
// stores ids[r] and drops the key; the key itself is known to every lane,
// and lane r keeps it (ranks from 32 on go through w[r]).  Afterwards each
// rank's lane computes its weight:
// p = expf(v - max) / sum over all E of expf(v - max) (each lane sums its
// experts in j order, then a fixed xor-shuffle tree);
// weight = p, or p / (sum of the k selected p, in rank order) when renorm.
// ids and w must be visible to the whole warp (shared or global memory).
template <int NPER, class Logit>
__device__ __forceinline__ void select_token_n(Logit lg, int E, int k, int renorm, int lane, int32_t *ids, float *w,
                                              float *sv) {
    (void)sv;
    constexpr uint32_t kAll = 0xffffffffu;
    uint32_t key[NPER];
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        key[j] = e < E ? logit_key(lg(e)) : 0u;
    }
    // this lane's best key, the lowest j among equal keys
    uint32_t bk = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (key[j] > bk) {
            bk = key[j];
            bj = j;
        }
    uint32_t mk = __reduce_max_sync(kAll, bk);
    const float m = key_logit(mk);
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (lane + 32 * j < E) z += expf(key_logit(key[j]) - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kAll, z, o);
    uint32_t rk = 0u;  // the key of rank `lane`
    for (int r = 0; r < k; ++r) {
        if (r > 0) mk = __reduce_max_sync(kAll, bk);
        const uint32_t held = __ballot_sync(kAll, bk == mk);
        int wl = __ffs(held) - 1;
        if (held & (held - 1u))  // a tie across lanes: the lowest expert index
            wl = (int)(__reduce_min_sync(kAll, bk == mk ? (uint32_t)(lane + 32 * bj) : 0xffffffffu) & 31u);
        if (lane == (r & 31)) {
            if (r < 32) rk = mk;
            else w[r] = __uint_as_float(mk);
        }
        if (lane == wl) {  // the winner records its expert, drops it and finds its next best
            ids[r] = lane + 32 * bj;
#pragma unroll
            for (int j = 0; j < NPER; ++j)
                if (j == bj) key[j] = 0u;
            bk = 0u;
            bj = 0;
#pragma unroll
            for (int j = 0; j < NPER; ++j)
                if (key[j] > bk) {
                    bk = key[j];
                    bj = j;
                }
        }
    }
    __syncwarp();
    float p = 0.f;  // rank `lane`'s weight
    if (lane < k) p = expf(key_logit(rk) - m) / z;
    for (int r = lane + 32; r < k; r += 32) w[r] = expf(key_logit(__float_as_uint(w[r])) - m) / z;
    if (renorm) {
        float psel = 0.f;
        const int k1 = k < 32 ? k : 32;
        for (int r = 0; r < k1; ++r) psel += __shfl_sync(kAll, p, r);
        __syncwarp();
        for (int r = 32; r < k; ++r) psel += w[r];
        __syncwarp();
        p = p / psel;
        for (int r = lane + 32; r < k; r += 32) w[r] = w[r] / psel;
    }
    if (lane < k) w[lane] = p;
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

// The same selection for logits in global memory (one token's row), kept out
// of line with two instances (up to 2 and up to 8 experts per lane): a kernel that selects
// once per launch keeps its hot loops close together in the instruction
// cache instead of carrying an unrolled copy per expert count.
static __device__ __noinline__ void select_token_global(const float *logits, int E, int k, int renorm, int lane,
                                                 int32_t *ids, float *w) {
    if (E <= 64)
        select_token_n<2>([&](int e) { return __ldcg(logits + e); }, E, k, renorm, lane, ids, w, nullptr);
    else
        select_token_n<8>([&](int e) { return __ldcg(logits + e); }, E, k, renorm, lane, ids, w, nullptr);
}
#endif  // __CUDACC__

}  // namespace spx
