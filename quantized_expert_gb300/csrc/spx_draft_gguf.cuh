// spx_draft_gguf.cuh -- the GGUF draft formats' arithmetic of one routed item
// of the draft launch (GGUF Q8_0, Q2_K and Q4_K experts; the gate/up items of
// a 16-column slice, the down items of a 32-output pair).  Included by
// spx_draft.cu only; the layouts are the repacked ones of spx_internal.cuh.
//
// Formats (GGUF, as the ai.info summary of the Specter paper reports GGUF
// drafts at Q2, Q4 and Q8 in its Main Findings):
//   Q8_0: W = d * code, one fp16 d per 32 input weights, int8 codes;
//   Q2_K: super-blocks of 256, W = d * sc * q - dmin * m, 4-bit sc and m per
//         sub-block of 16, 2-bit q;
//   Q4_K: super-blocks of 256, W = d * sc * q - dmin * m, 6-bit sc and m per
//         sub-block of 32, 4-bit q.
#pragma once
#include "spx_internal.cuh"

namespace spx {

// Gate/up item, Q8_0: groups [k0, k0+n) of 128 rows.  run[t][*] gathers tile
// t's accumulators (rows g, g+8; token columns 2*q4, 2*q4+1); xr is this
// lane's activation row (token g) in shared memory, okx whether it is real.
template <int NTW>
__device__ __forceinline__ void gguf_rg_q8(float (&run)[NTW][4], const uint8_t *stage, int k0, int n,
                                           const __half *xr, bool okx, int lane) {
    const int g = lane >> 2;
    // GGUF Q8_0: per group of 128 rows, four blocks of 32 rows (two
    // k-steps) with their own scales; the codes become exact fp16
    // values, one block's products are summed, then scaled
    for (int gr = 0; gr < n; ++gr) {
        const uint8_t *gp = stage + (size_t)gr * kQ8GroupBytes;
        const __half *scp = reinterpret_cast<const __half *>(gp);
#pragma unroll
        for (int sb = 0; sb < 4; ++sb) {
            float acc[NTW][4] = {};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int kl = 2 * sb + kk;
                const int ks = (k0 + gr) * 8 + kl;
                const uint4 v = lds128(gp + kQ8ScaleBytes + kl * 512 + lane * 16);
                const uint32_t b0 = okx ? lds32(xr + 16 * ks) : 0u;
                const uint32_t b1 = okx ? lds32(xr + 16 * ks + 8) : 0u;
                uint32_t a[4];
                q8_frag(v.x, v.y, a);
                mma_16816(acc[0], a, b0, b1);
                q8_frag(v.z, v.w, a);
                mma_16816(acc[1], a, b0, b1);
            }
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                const float sa = __half2float(scp[sb * 32 + t * 16 + g]);
                const float sc = __half2float(scp[sb * 32 + t * 16 + g + 8]);
                run[t][0] = fmaf(sa, acc[t][0], run[t][0]);
                run[t][1] = fmaf(sa, acc[t][1], run[t][1]);
                run[t][2] = fmaf(sc, acc[t][2], run[t][2]);
                run[t][3] = fmaf(sc, acc[t][3], run[t][3]);
            }
        }
    }
}

// Gate/up item, Q2_K: super-blocks [k0, k0+n) of 256 rows; sxh / sxl hold the
// token's sums of x over 16 rows (fp16 hi and lo parts, [H/16] each).
template <int NTW>
__device__ __forceinline__ void gguf_rg_q2k(float (&run)[NTW][4], const uint8_t *stage, int k0, int n,
                                            const __half *xr, bool okx, int lane, const __half *sxh,
                                            const __half *sxl) {
    const int g = lane >> 2, q4 = lane & 3;
    // GGUF Q2_K: super-blocks of 256 rows = 16 k-steps; k-step b is
    // sub-block b of every row, with its own 4-bit scale sc and min m.
    // The fragment holds sc*q (exact in fp16: one fused multiply-add
    // of the magic value 1024 + q), so one accumulator spans the
    // super-block; the mins enter through one more product, of the
    // rows' 16 mins with the token's 16 sub-block sums of x (those
    // split into an fp16 pair hi + lo).  Then d and dmin per row.
    const __half2 k1024 = u32_as_h2(0x64006400u), km1024 = u32_as_h2(0xE400E400u);
    for (int gr = 0; gr < n; ++gr) {
        const uint8_t *sp = stage + (size_t)gr * kQ2kSbBytes;
        const __half *dd = reinterpret_cast<const __half *>(sp);  // d [32], then dmin [32]
        const int sbg = k0 + gr;                                // super-block of H
        const uint4 c0 = lds128(sp + kQ2kScaleOff + g * 32);
        const uint4 c1 = lds128(sp + kQ2kScaleOff + g * 32 + 16);
        const uint32_t scw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        float am[NTW][4] = {}, an[NTW][4] = {};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 v = lds128(sp + kQ2kCodeOff + c * 512 + lane * 16);
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int kl = 4 * c + kk;
                const int ks = sbg * 16 + kl;
                const uint32_t b0 = okx ? lds32(xr + 16 * ks) : 0u;
                const uint32_t b1 = okx ? lds32(xr + 16 * ks + 8) : 0u;
                // the k-step's four scale nibbles (t, row g / g+8), in both halves
                const uint32_t su = ((scw[kl >> 1] >> (16 * (kl & 1))) & 0xFFFFu) * 0x10001u;
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    const __half2 sa2 =
                        __hsub2(u32_as_h2(lop3_and_or(su >> (8 * t), 0x000F000Fu, 0x64006400u)), k1024);
                    const __half2 sb2 =
                        __hsub2(u32_as_h2(lop3_and_or(su >> (8 * t + 4), 0x000F000Fu, 0x64006400u)), k1024);
                    const __half2 oa2 = __hmul2(sa2, km1024), ob2 = __hmul2(sb2, km1024);
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t raw =
                            lop3_and_or(words[kk] >> (2 * (4 * t + r)), 0x00030003u, 0x64006400u);
                        a[r] = h2_as_u32(__hfma2(u32_as_h2(raw), (r & 1) ? sb2 : sa2, (r & 1) ? ob2 : oa2));
                    }
                    mma_16816(am[t], a, b0, b1);
                }
            }
        }
        const uint32_t bh0 = okx ? lds32(sxh + sbg * 16 + 2 * q4) : 0u;
        const uint32_t bh1 = okx ? lds32(sxh + sbg * 16 + 2 * q4 + 8) : 0u;
        const uint32_t bl0 = okx ? lds32(sxl + sbg * 16 + 2 * q4) : 0u;
        const uint32_t bl1 = okx ? lds32(sxl + sbg * 16 + 2 * q4 + 8) : 0u;
        const uint2 mw = lds64(sp + kQ2kMinOff + lane * 8);
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
            const uint32_t w = t == 0 ? mw.x : mw.y;
            uint32_t a[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                a[r] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w >> (4 * r), 0x000F000Fu, 0x64006400u)), k1024));
            mma_16816(an[t], a, bh0, bh1);
            mma_16816(an[t], a, bl0, bl1);
        }
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
            const float da = __half2float(dd[t * 16 + g]), db = __half2float(dd[t * 16 + g + 8]);
            const float ma = __half2float(dd[32 + t * 16 + g]), mb = __half2float(dd[32 + t * 16 + g + 8]);
            run[t][0] += da * am[t][0] - ma * an[t][0];
            run[t][1] += da * am[t][1] - ma * an[t][1];
            run[t][2] += db * am[t][2] - mb * an[t][2];
            run[t][3] += db * am[t][3] - mb * an[t][3];
        }
    }
}

// Gate/up item, Q4_K: super-blocks [k0, k0+n) of 256 rows; sxh / sxl hold the
// token's sums of x over 32 rows (fp16 hi and lo parts, [H/32] each).
template <int NTW>
__device__ __forceinline__ void gguf_rg_q4k(float (&run)[NTW][4], const uint8_t *stage, int k0, int n,
                                            const __half *xr, bool okx, int lane, const __half *sxh,
                                            const __half *sxl) {
    const int g = lane >> 2, q4 = lane & 3;
    // GGUF Q4_K: super-blocks of 256 rows; sub-block c = 32 rows = k-steps
    // 2c and 2c+1, with a 6-bit scale and min per row.  As for Q2_K the
    // fragment holds scale*q (<= 945, exact in fp16 through one fused
    // multiply-add), and the mins enter through one more product with the
    // token's eight 32-row sums of x (k = sub-block, k >= 8 zero).
    const __half2 k1024 = u32_as_h2(0x64006400u), km1024 = u32_as_h2(0xE400E400u);
    const uint32_t kExp = 0x64646464u;
    for (int gr = 0; gr < n; ++gr) {
        const uint8_t *sp = stage + (size_t)gr * kQ4kSbBytes;
        const __half *dd = reinterpret_cast<const __half *>(sp);  // d [32], then dmin [32]
        const int sbg = k0 + gr;                                // super-block of H
        const uint4 c0 = lds128(sp + kQ4kScaleOff + g * 32);
        const uint4 c1 = lds128(sp + kQ4kScaleOff + g * 32 + 16);
        const uint32_t scw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        float am[NTW][4] = {}, an[NTW][4] = {};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = lds128(sp + kQ4kCodeOff + c * 512 + lane * 16);
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};  // [k-step][tile]
            __half2 sc2[NTW][2], of2[NTW][2];                 // (scale, -1024 scale) of rows g, g+8
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t sel = (2 * t + j) * 0x0101u + 0x4040u;  // byte 2t+j under 0x64
                    sc2[t][j] = __hsub2(u32_as_h2(__byte_perm(scw[c], kExp, sel)), k1024);
                    of2[t][j] = __hmul2(sc2[t][j], km1024);
                }
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int ks = sbg * 16 + 2 * c + kk;
                const uint32_t b0 = okx ? lds32(xr + 16 * ks) : 0u;
                const uint32_t b1 = okx ? lds32(xr + 16 * ks + 8) : 0u;
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    const uint32_t w = words[2 * kk + t];
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t raw = lop3_and_or(w >> (4 * r), 0x000F000Fu, 0x64006400u);
                        a[r] = h2_as_u32(__hfma2(u32_as_h2(raw), sc2[t][r & 1], of2[t][r & 1]));
                    }
                    mma_16816(am[t], a, b0, b1);
                }
            }
        }
        const uint32_t bh0 = okx ? lds32(sxh + sbg * 8 + 2 * q4) : 0u;
        const uint32_t bl0 = okx ? lds32(sxl + sbg * 8 + 2 * q4) : 0u;
        const uint2 mw = lds64(sp + kQ4kMinOff + lane * 8);
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
            const uint32_t w = t == 0 ? mw.x : mw.y;
            uint32_t a[4];
            a[0] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, kExp, 0x4140u)), k1024));
            a[1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, kExp, 0x4342u)), k1024));
            a[2] = 0u;
            a[3] = 0u;
            mma_16816(an[t], a, bh0, 0u);
            mma_16816(an[t], a, bl0, 0u);
        }
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
            const float da = __half2float(dd[t * 16 + g]), db = __half2float(dd[t * 16 + g + 8]);
            const float ma = __half2float(dd[32 + t * 16 + g]), mb = __half2float(dd[32 + t * 16 + g + 8]);
            run[t][0] += da * am[t][0] - ma * an[t][0];
            run[t][1] += da * am[t][1] - ma * an[t][1];
            run[t][2] += db * am[t][2] - mb * an[t][2];
            run[t][3] += db * am[t][3] - mb * an[t][3];
        }
    }
}

// Down item, Q8_0 (every GGUF format): groups [0, n) of 128 rows of the item's
// range of I; hsl holds the range's intermediate h (B fragments, [k-step][T]).
__device__ __forceinline__ void gguf_rd_q8(float (&run)[2][4], const uint8_t *stage, int n, const uint2 *hsl,
                                           int T, bool okb, int lane) {
    const int g = lane >> 2, q4 = lane & 3;
    // GGUF Q8_0, as the gate/up items: four 32-row blocks per group
    for (int gr = 0; gr < n; ++gr) {
        const uint8_t *gp = stage + (size_t)gr * kQ8GroupBytes;
        const __half *scp = reinterpret_cast<const __half *>(gp);
#pragma unroll
        for (int sb = 0; sb < 4; ++sb) {
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int kl = 2 * sb + kk;
                const int ksr = gr * 8 + kl;  // k-step within the slice
                const uint4 v = lds128(gp + kQ8ScaleBytes + kl * 512 + lane * 16);
                uint2 bv = make_uint2(0u, 0u);
                if (okb) bv = *reinterpret_cast<const uint2 *>(hsl + ((size_t)ksr * T + g) * 4 + q4);
                uint32_t a[4];
                q8_frag(v.x, v.y, a);
                mma_16816(acc[0], a, bv.x, bv.y);
                q8_frag(v.z, v.w, a);
                mma_16816(acc[1], a, bv.x, bv.y);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float sa = __half2float(scp[sb * 32 + q * 16 + g]);
                const float sc = __half2float(scp[sb * 32 + q * 16 + g + 8]);
                run[q][0] = fmaf(sa, acc[q][0], run[q][0]);
                run[q][1] = fmaf(sa, acc[q][1], run[q][1]);
                run[q][2] = fmaf(sc, acc[q][2], run[q][2]);
                run[q][3] = fmaf(sc, acc[q][3], run[q][3]);
            }
        }
    }
}

// The x sums the K-quant gate/up items use: called by every lane of a warp
// with `sum`, this lane's sum of the 8 activations of chunk `idx` ([t][H/8]);
// Q2_K stores sums over 16 rows at sx[t][H/16], Q4_K over 32 rows at
// sx[t][H/32], each as an fp16 pair: hi, then lo (T rows further on).
template <bool Q2K, bool Q4K>
__device__ __forceinline__ void kquant_x_sums(float sum, int lane, int idx, int T, int H, __half *sx) {
    if constexpr (Q2K) {  // this lane's chunk and its pair's
        const float s16 = sum + __shfl_xor_sync(0xffffffffu, sum, 1);
        if ((lane & 1) == 0 && idx < T * (H / 8)) {
            const __half hi = __float2half_rn(s16);
            sx[idx / 2] = hi;  // [t][16-row block]: idx/2 = t*(H/16) + block
            sx[T * (H / 16) + idx / 2] = __float2half_rn(s16 - __half2float(hi));
        }
    }
    if constexpr (Q4K) {  // four chunks
        float s32 = sum + __shfl_xor_sync(0xffffffffu, sum, 1);
        s32 += __shfl_xor_sync(0xffffffffu, s32, 2);
        if ((lane & 3) == 0 && idx < T * (H / 8)) {
            const __half hi = __float2half_rn(s32);
            sx[idx / 4] = hi;  // [t][32-row block]: idx/4 = t*(H/32) + block
            sx[T * (H / 32) + idx / 4] = __float2half_rn(s32 - __half2float(hi));
        }
    }
}

}  // namespace spx
