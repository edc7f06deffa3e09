// spx_pack.cu -- one-time repack of canonical expert tensors into the packed
// units the expert launch streams (see spx_internal.cuh for the geometry).
//
// Canonical inputs: GPTQ INT4 with group size 128 and zero point 8 (richland.au
// post, "What shipped"): qweight [K/8][N] int32 with code kk at bits
// 4*(kk%8), scales [K/128][N] fp16; FP16 experts in PyTorch [out][in] layout.
// The repack is a pure permutation of codes / values (scales are copied), so
// it is bit-exact and deterministic.
#include "spx_internal.cuh"

namespace spx {

__device__ __forceinline__ uint32_t gptq_code(const int32_t *q, int N, int kk, int n) {
    const uint32_t w = static_cast<uint32_t>(q[(size_t)(kk >> 3) * N + n]);
    return (w >> (4 * (kk & 7))) & 15u;
}

// Gate/up section: H/128 groups, each = 2S fp16 scales (gate columns then up
// columns) followed by 8 k-steps of codes in blocks of KB = 2/MS k-steps
// (32 lanes x 16 B; lane word w = [ki][tile], tile t < MS gate columns
// 16t.., t >= MS up columns 16(t-MS)..; nibble j of a word is fragment
// register (j & 3), half (j >> 2)).
__global__ void w4_pack_scales(const uint16_t *s_gate, const uint16_t *s_up, int E, int H, int I, int S,
                               uint8_t *packed) {
    const int spe = I / S, G = H / 128;
    const size_t total = (size_t)E * spe * G * 2 * S;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int c2 = idx % (2 * S);
        const int grp = (idx / (2 * S)) % G;
        const size_t unit = idx / ((size_t)2 * S * G);
        const int e = unit / spe, j = unit % spe;
        const int i = j * S + (c2 % S);
        const uint16_t *src = c2 < S ? s_gate : s_up;
        uint16_t *dst = reinterpret_cast<uint16_t *>(packed + unit * w4_unit_bytes(H, S) + grp * w4_group_bytes(S));
        dst[c2] = src[((size_t)e * G + grp) * I + i];
    }
}

__global__ void w4_pack_gu(const int32_t *qg, const int32_t *qu, int E, int H, int I, int S, uint8_t *packed) {
    const int MS = S / 16, KB = 2 / MS, NTILE = 2 * MS, spe = I / S;
    const int nblk = (H / 16) / KB;  // blocks per unit
    const int bpg = 8 / KB;          // blocks per group
    const size_t total = (size_t)E * spe * nblk * 32 * 4;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int wi = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int b = (idx >> 7) % nblk;
        const size_t unit = (idx >> 7) / nblk;
        const int e = unit / spe, jsl = unit % spe;
        const int ki = wi / NTILE, t = wi % NTILE;
        const int ks = b * KB + ki;
        const int32_t *q = (t < MS ? qg : qu) + (size_t)e * (H / 8) * I;
        const int icol0 = jsl * S + 16 * (t % MS);
        uint32_t word = 0;
        for (int nib = 0; nib < 8; ++nib) {
            const int r = nib & 3, hh = nib >> 2;
            const int m = frag_row(lane, r), kc = frag_col(lane, r, hh);
            word |= gptq_code(q, I, 16 * ks + kc, icol0 + m) << (4 * nib);
        }
        const int grp = b / bpg, ib = b % bpg;
        uint8_t *gbase = packed + unit * w4_unit_bytes(H, S) + grp * w4_group_bytes(S) + 4 * S;
        reinterpret_cast<uint32_t *>(gbase + ib * 512)[lane * 4 + wi] = word;
    }
}

// Down codes: block b holds MB = 4/MS m-tiles; lane word w = [tile_in][ks];
// A[m][kc] = code of W_down[i0 + 16 ks + kc][down_col(mt, m)].
__global__ void w4_pack_down(const int32_t *qd, int E, int H, int I, int S, uint8_t *packed) {
    const int MS = S / 16, MB = 4 / MS, spe = I / S;
    const int nblk = (H / 16) / MB;
    const size_t total = (size_t)E * spe * nblk * 32 * 4;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int wi = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int b = (idx >> 7) % nblk;
        const size_t unit = (idx >> 7) / nblk;
        const int e = unit / spe, jsl = unit % spe;
        const int tin = wi / MS, ks = wi % MS;
        const int mt = b * MB + tin;
        const int32_t *q = qd + (size_t)e * (I / 8) * H;
        uint32_t word = 0;
        for (int nib = 0; nib < 8; ++nib) {
            const int r = nib & 3, hh = nib >> 2;
            const int m = frag_row(lane, r), kc = frag_col(lane, r, hh);
            word |= gptq_code(q, H, jsl * S + 16 * ks + kc, down_col(mt, m)) << (4 * nib);
        }
        uint32_t *dst = reinterpret_cast<uint32_t *>(packed + unit * w4_unit_bytes(H, S) + w4_gu_bytes(H, S));
        dst[(size_t)b * 128 + lane * 4 + wi] = word;
    }
}

// FP16 gate/up: block = k-step ks: [tile t (0 gate, 1 up)][lane] x 16 B; the
// 16 B are the fragment registers r = 0..3, halves h = 0..1.
__global__ void f16_pack_gu(const uint16_t *wg, const uint16_t *wu, int E, int H, int I, uint8_t *packed) {
    const int spe = I / kF16S;
    const size_t total = (size_t)E * spe * (H / 16) * 2 * 32 * 4;  // 32-bit words
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int r = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int t = (idx >> 7) & 1;
        const int ks = (idx >> 8) % (H / 16);
        const size_t unit = (idx >> 8) / (H / 16);
        const int e = unit / spe, jsl = unit % spe;
        const uint16_t *w = (t == 0 ? wg : wu) + (size_t)e * I * H;
        const int i = jsl * kF16S + frag_row(lane, r);
        uint32_t word = 0;
        for (int hh = 0; hh < 2; ++hh) {
            const int kk = 16 * ks + frag_col(lane, r, hh);
            word |= (uint32_t)w[(size_t)i * H + kk] << (16 * hh);
        }
        uint32_t *dst = reinterpret_cast<uint32_t *>(packed + unit * f16_unit_bytes(H));
        dst[(((size_t)ks * 2 + t) * 32 + lane) * 4 + r] = word;
    }
}

// FP16 down: block = m-tile pair P: [q][lane] x 16 B; A[m][kc] =
// W_down[down_col(2P+q, m)][i0 + kc].
__global__ void f16_pack_down(const uint16_t *wd, int E, int H, int I, uint8_t *packed) {
    const int spe = I / kF16S;
    const size_t total = (size_t)E * spe * (H / 32) * 2 * 32 * 4;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int r = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int q = (idx >> 7) & 1;
        const int P = (idx >> 8) % (H / 32);
        const size_t unit = (idx >> 8) / (H / 32);
        const int e = unit / spe, jsl = unit % spe;
        const uint16_t *w = wd + (size_t)e * H * I;
        const int n = down_col(2 * P + q, frag_row(lane, r));
        uint32_t word = 0;
        for (int hh = 0; hh < 2; ++hh) {
            const int i = jsl * kF16S + frag_col(lane, r, hh);
            word |= (uint32_t)w[(size_t)n * I + i] << (16 * hh);
        }
        uint32_t *dst = reinterpret_cast<uint32_t *>(packed + unit * f16_unit_bytes(H) + f16_gu_bytes(H));
        dst[(((size_t)P * 2 + q) * 32 + lane) * 4 + r] = word;
    }
}

// INT4 down, column-block-major: scales of (e, pair Q, group grp).
__global__ void w4_pack_colblk_scales(const uint16_t *s_down, int E, int H, int I, uint8_t *region) {
    const int NQ = H / 32, G = I / 128;
    const size_t total = (size_t)E * NQ * G * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int qm = idx % 32;
        const size_t gi = idx / 32;  // (e * NQ + Q) * G + grp
        const int grp = gi % G;
        const int Q = (gi / G) % NQ;
        const int e = gi / ((size_t)G * NQ);
        const int n = down_col(2 * Q + (qm >> 4), qm & 15);
        uint16_t *dst = reinterpret_cast<uint16_t *>(region + gi * kW4ColGroupBytes);
        dst[qm] = s_down[((size_t)e * G + grp) * H + n];
    }
}

// INT4 down, column-block-major: codes; block ib of a group holds k-steps
// 8*grp + 2*ib + {0,1}; lane word w = [ks_in][tile].
__global__ void w4_pack_colblk_codes(const int32_t *qd, int E, int H, int I, uint8_t *region) {
    const int NQ = H / 32, G = I / 128;
    const size_t total = (size_t)E * NQ * G * 4 * 128;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int wi = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int ib = (idx >> 7) & 3;
        const size_t gi = idx >> 9;  // (e * NQ + Q) * G + grp
        const int grp = gi % G;
        const int Q = (gi / G) % NQ;
        const int e = gi / ((size_t)G * NQ);
        const int ks = grp * 8 + ib * 2 + (wi >> 1);
        const int q = wi & 1;
        const int32_t *qe = qd + (size_t)e * (I / 8) * H;
        uint32_t word = 0;
        for (int nib = 0; nib < 8; ++nib) {
            const int r = nib & 3, hh = nib >> 2;
            const int m = frag_row(lane, r), kc = frag_col(lane, r, hh);
            word |= gptq_code(qe, H, 16 * ks + kc, down_col(2 * Q + q, m)) << (4 * nib);
        }
        reinterpret_cast<uint32_t *>(region + gi * kW4ColGroupBytes + 64 + ib * 512)[lane * 4 + wi] = word;
    }
}

// Shared expert down, pair-major: [P][ks][tile q][lane] x 16 B;
// A[m][kc] = W_down[down_col(2P+q, m)][16 ks + kc].
__global__ void f16_pack_pairdown(const uint16_t *wd, int H, int I, uint8_t *region) {
    const int NP = H / 32, NK = I / 16;
    const size_t total = (size_t)NP * NK * 2 * 32 * 4;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int r = idx & 3;
        const int lane = (idx >> 2) & 31;
        const int q = (idx >> 7) & 1;
        const size_t pk = idx >> 8;  // P * NK + ks
        const int ks = pk % NK, P = pk / NK;
        const int n = down_col(2 * P + q, frag_row(lane, r));
        uint32_t word = 0;
        for (int hh = 0; hh < 2; ++hh) word |= (uint32_t)wd[(size_t)n * I + 16 * ks + frag_col(lane, r, hh)] << (16 * hh);
        reinterpret_cast<uint32_t *>(region)[((pk * 2 + q) * 32 + lane) * 4 + r] = word;
    }
}

static int grid_for(size_t total) {
    size_t g = (total + 255) / 256;
    if (g > 65535) g = 65535;
    if (g < 1) g = 1;
    return (int)g;
}

// Zero points, gate/up: [E][I/S units][H/128 groups][2S] fp16 in the order
// of the packed scales (gate columns, then up columns).
__global__ void w4_pack_zeros_gu(const int32_t *zg, const int32_t *zu, int E, int H, int I, int S, uint16_t *dst) {
    const int spe = I / S, G = H / 128;
    const size_t total = (size_t)E * spe * G * 2 * S;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int c2 = idx % (2 * S);
        const int grp = (idx / (2 * S)) % G;
        const size_t unit = idx / ((size_t)2 * S * G);
        const int e = unit / spe, j = unit % spe;
        const int i = j * S + (c2 % S);
        const int32_t *src = c2 < S ? zg : zu;
        const uint32_t w = static_cast<uint32_t>(src[((size_t)e * G + grp) * (I / 8) + i / 8]);
        dst[idx] = __half_as_ushort(__float2half((float)((w >> (4 * (i % 8))) & 15u)));
    }
}

// Zero points, down: [E][H/32 pairs][I/128 groups][32] fp16 in the order of
// the column-block scales.
__global__ void w4_pack_zeros_dn(const int32_t *zd, int E, int H, int I, uint16_t *dst) {
    const int NQ = H / 32, G = I / 128;
    const size_t total = (size_t)E * NQ * G * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int qm = idx % 32;
        const size_t gi = idx / 32;
        const int grp = gi % G;
        const int Q = (gi / G) % NQ;
        const int e = gi / ((size_t)G * NQ);
        const int n = down_col(2 * Q + (qm >> 4), qm & 15);
        const uint32_t w = static_cast<uint32_t>(zd[((size_t)e * G + grp) * (H / 8) + n / 8]);
        dst[idx] = __half_as_ushort(__float2half((float)((w >> (4 * (n % 8))) & 15u)));
    }
}

// ---------------------------------------------------------- GGUF Q8_0 --
// Canonical Q8_0 matrix [out N][in K]: per row, K/32 blocks of 34 bytes (fp16
// scale, little-endian, then 32 int8 codes).  Code and scale of (n, k):
__device__ __forceinline__ uint8_t q8_code(const uint8_t *w, int K, size_t e, int N, int n, int k) {
    return w[((e * N + n) * (K / 32) + k / 32) * 34 + 2 + k % 32];
}
__device__ __forceinline__ uint16_t q8_scale(const uint8_t *w, int K, size_t e, int N, int n, int blk) {
    const uint8_t *b = w + ((e * N + n) * (K / 32) + blk) * 34;
    return (uint16_t)(b[0] | (b[1] << 8));
}

// Gate/up units: one thread per (unit, group, k-step, lane, tile) writes the
// lane's 8 codes of that tile; scales: one thread per (unit, group, block, column).
__global__ void q8_pack_gu(const uint8_t *wg, const uint8_t *wu, int E, int H, int I, uint8_t *packed) {
    const int spe = I / 16, G = H / 128;
    const size_t total = (size_t)E * spe * G * 8 * 32 * 2;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(idx & 1);
        const int lane = (int)((idx >> 1) & 31);
        const int kl = (int)((idx >> 6) & 7);
        const size_t ug = idx >> 9;  // unit * G + group
        const int grp = (int)(ug % G);
        const size_t unit = ug / G;
        const size_t e = unit / spe;
        const int j = (int)(unit % spe);
        const uint8_t *src = t == 0 ? wg : wu;
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int jb = 0; jb < 8; ++jb) {
            const int r = jb >> 1;
            const int n = j * 16 + frag_row(lane, r);
            const int k = grp * 128 + kl * 16 + frag_col(lane, r, jb & 1);
            w[jb >> 2] |= (uint32_t)q8_code(src, H, e, I, n, k) << (8 * (jb & 3));
        }
        uint8_t *dst = packed + unit * q8_unit_bytes(H) + (size_t)grp * kQ8GroupBytes + kQ8ScaleBytes + kl * 512 +
                       lane * 16 + t * 8;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    }
    const size_t ns = (size_t)E * spe * G * 4 * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < ns; idx += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx & 31);
        const int sb = (int)((idx >> 5) & 3);
        const size_t ug = idx >> 7;
        const int grp = (int)(ug % G);
        const size_t unit = ug / G;
        const size_t e = unit / spe;
        const int n = (int)(unit % spe) * 16 + (c & 15);
        const uint16_t v = q8_scale(c < 16 ? wg : wu, H, e, I, n, grp * 4 + sb);
        reinterpret_cast<uint16_t *>(packed + unit * q8_unit_bytes(H) + (size_t)grp * kQ8GroupBytes)[sb * 32 + c] = v;
    }
}

// Down, column-block-major: one thread per (expert, pair, group, k-step, lane,
// tile) for the codes, one per (expert, pair, group, block, tile row) for scales.
__global__ void q8_pack_dn(const uint8_t *wd, int E, int H, int I, uint8_t *region) {
    const int NQ = H / 32, G = I / 128;
    const size_t total = (size_t)E * NQ * G * 8 * 32 * 2;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(idx & 1);
        const int lane = (int)((idx >> 1) & 31);
        const int kl = (int)((idx >> 6) & 7);
        const size_t gi = idx >> 9;  // (e * NQ + Q) * G + group
        const int grp = (int)(gi % G);
        const int Q = (int)((gi / G) % NQ);
        const size_t e = gi / ((size_t)G * NQ);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int jb = 0; jb < 8; ++jb) {
            const int r = jb >> 1;
            const int n = down_col(2 * Q + q, frag_row(lane, r));
            const int i = grp * 128 + kl * 16 + frag_col(lane, r, jb & 1);
            w[jb >> 2] |= (uint32_t)q8_code(wd, I, e, H, n, i) << (8 * (jb & 3));
        }
        uint8_t *dst = region + gi * kQ8GroupBytes + kQ8ScaleBytes + kl * 512 + lane * 16 + q * 8;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    }
    const size_t ns = (size_t)E * NQ * G * 4 * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < ns; idx += (size_t)gridDim.x * blockDim.x) {
        const int qm = (int)(idx & 31);
        const int sb = (int)((idx >> 5) & 3);
        const size_t gi = idx >> 7;
        const int grp = (int)(gi % G);
        const int Q = (int)((gi / G) % NQ);
        const size_t e = gi / ((size_t)G * NQ);
        const int n = down_col(2 * Q + (qm >> 4), qm & 15);
        reinterpret_cast<uint16_t *>(region + gi * kQ8GroupBytes)[sb * 32 + qm] = q8_scale(wd, I, e, H, n, grp * 4 + sb);
    }
}

// ---------------------------------------------------------- GGUF Q2_K --
// Canonical Q2_K matrix [out N][in K]: per row, K/256 super-blocks of 84
// bytes (16 sub-block bytes: scale low nibble, min high nibble; 64 code bytes;
// fp16 d; fp16 dmin).  Code of value wi (0..255) of a super-block:
__device__ __forceinline__ const uint8_t *q2k_block(const uint8_t *w, int K, size_t e, int N, int n, int sb) {
    return w + ((e * N + n) * (K / 256) + sb) * 84;
}
__device__ __forceinline__ uint32_t q2k_code(const uint8_t *blk, int wi) {
    return (blk[16 + 32 * (wi / 128) + wi % 32] >> (2 * ((wi % 128) / 32))) & 3u;
}

// Gate/up units: codes, one thread per (unit, super-block, code block, lane,
// k-step word); then d/dmin, sub-block scale words and min words.
__global__ void q2k_pack_gu(const uint8_t *wg, const uint8_t *wu, int E, int H, int I, uint8_t *packed) {
    const int spe = I / 16, NS = H / 256;
    const size_t npair = (size_t)E * spe * NS;
    const size_t ub = q2k_unit_bytes(H);
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < npair * 512;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int kk = (int)(idx & 3);
        const int lane = (int)((idx >> 2) & 31);
        const int c = (int)((idx >> 7) & 3);
        const size_t us = idx >> 9;  // unit * NS + super-block
        const int sb = (int)(us % NS);
        const size_t unit = us / NS;
        const size_t e = unit / spe;
        const int jj = (int)(unit % spe);
        uint32_t word = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint8_t *blk = q2k_block(t ? wu : wg, H, e, I, jj * 16 + frag_row(lane, r), sb);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    word |= q2k_code(blk, 16 * (4 * c + kk) + frag_col(lane, r, h)) << (16 * h + 2 * (4 * t + r));
            }
        }
        *reinterpret_cast<uint32_t *>(packed + unit * ub + (size_t)sb * kQ2kSbBytes + kQ2kCodeOff + c * 512 +
                                      lane * 16 + kk * 4) = word;
    }
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < npair * 224;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int item = (int)(idx % 224);
        const size_t us = idx / 224;
        const int sb = (int)(us % NS);
        const size_t unit = us / NS;
        const size_t e = unit / spe;
        const int jj = (int)(unit % spe);
        uint8_t *base = packed + unit * ub + (size_t)sb * kQ2kSbBytes;
        if (item < 32) {  // d and dmin of tile item/16, row item%16
            const uint8_t *blk = q2k_block(item < 16 ? wg : wu, H, e, I, jj * 16 + item % 16, sb);
            reinterpret_cast<uint16_t *>(base)[item] = (uint16_t)(blk[80] | (blk[81] << 8));
            reinterpret_cast<uint16_t *>(base)[32 + item] = (uint16_t)(blk[82] | (blk[83] << 8));
        } else if (item < 160) {  // scale nibbles of (g, k-step)
            const int g = (item - 32) / 16, ks = (item - 32) % 16;
            uint32_t u = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint8_t *blk = q2k_block(j >> 1 ? wu : wg, H, e, I, jj * 16 + g + 8 * (j & 1), sb);
                u |= (uint32_t)(blk[ks] & 15) << (4 * j);
            }
            reinterpret_cast<uint16_t *>(base + kQ2kScaleOff)[g * 16 + ks] = (uint16_t)u;
        } else {  // min nibbles of (lane, tile) in A-fragment order
            const int lane = (item - 160) / 2, t = (item - 160) % 2;
            uint32_t w = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint8_t *blk = q2k_block(t ? wu : wg, H, e, I, jj * 16 + frag_row(lane, r), sb);
#pragma unroll
                for (int h = 0; h < 2; ++h) w |= (uint32_t)(blk[frag_col(lane, r, h)] >> 4) << (16 * h + 4 * r);
            }
            reinterpret_cast<uint32_t *>(base + kQ2kMinOff)[lane * 2 + t] = w;
        }
    }
}

// ---------------------------------------------------------- GGUF Q4_K --
// Canonical Q4_K matrix [out N][in K]: per row, K/256 super-blocks of 144
// bytes (fp16 d, fp16 dmin, 12 bytes of 6-bit sub-block scales and mins, 128
// bytes of 4-bit codes).
__device__ __forceinline__ const uint8_t *q4k_block(const uint8_t *w, int K, size_t e, int N, int n, int sb) {
    return w + ((e * N + n) * (K / 256) + sb) * 144;
}
// 6-bit scale (want_min = 0) or min (1) of sub-block s (0..7): the first four
// sub-blocks keep theirs in the low 6 bits of bytes s / s+4; the last four
// take 4 bits from byte s+4 (scale low nibble, min high nibble) and their top
// 2 bits from the high bits of bytes s-4 (scale) / s (min).
__device__ __forceinline__ uint32_t q4k_param(const uint8_t *blk, int s, int want_min) {
    const uint8_t *b = blk + 4;
    if (s < 4) return (uint32_t)(b[s + 4 * want_min] & 63);
    if (!want_min) return (uint32_t)((b[s + 4] & 15) | ((b[s - 4] >> 6) << 4));
    return (uint32_t)((b[s + 4] >> 4) | ((b[s] >> 6) << 4));
}
__device__ __forceinline__ uint32_t q4k_code(const uint8_t *blk, int wi) {
    const uint8_t byte = blk[16 + 32 * (wi / 64) + wi % 32];
    return (wi % 64) < 32 ? (byte & 15u) : (uint32_t)(byte >> 4);
}

// Gate/up units: codes, one thread per (unit, super-block, block of 2
// k-steps, lane, word); then d/dmin, scale words and min words.
__global__ void q4k_pack_gu(const uint8_t *wg, const uint8_t *wu, int E, int H, int I, uint8_t *packed) {
    const int spe = I / 16, NS = H / 256;
    const size_t npair = (size_t)E * spe * NS;
    const size_t ub = q4k_unit_bytes(H);
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < npair * 1024;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int wd = (int)(idx & 3);  // lane word: k-step wd/2 of the block, tile wd%2
        const int lane = (int)((idx >> 2) & 31);
        const int c = (int)((idx >> 7) & 7);
        const size_t us = idx >> 10;  // unit * NS + super-block
        const int sb = (int)(us % NS);
        const size_t unit = us / NS;
        const size_t e = unit / spe;
        const int jj = (int)(unit % spe);
        const int t = wd & 1, ks = 2 * c + (wd >> 1);
        uint32_t word = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint8_t *blk = q4k_block(t ? wu : wg, H, e, I, jj * 16 + frag_row(lane, r), sb);
#pragma unroll
            for (int h = 0; h < 2; ++h) word |= q4k_code(blk, 16 * ks + frag_col(lane, r, h)) << (16 * h + 4 * r);
        }
        *reinterpret_cast<uint32_t *>(packed + unit * ub + (size_t)sb * kQ4kSbBytes + kQ4kCodeOff + c * 512 +
                                      lane * 16 + wd * 4) = word;
    }
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < npair * 160;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int item = (int)(idx % 160);
        const size_t us = idx / 160;
        const int sb = (int)(us % NS);
        const size_t unit = us / NS;
        const size_t e = unit / spe;
        const int jj = (int)(unit % spe);
        uint8_t *base = packed + unit * ub + (size_t)sb * kQ4kSbBytes;
        if (item < 32) {  // d and dmin of tile item/16, row item%16
            const uint8_t *blk = q4k_block(item < 16 ? wg : wu, H, e, I, jj * 16 + item % 16, sb);
            reinterpret_cast<uint16_t *>(base)[item] = (uint16_t)(blk[0] | (blk[1] << 8));
            reinterpret_cast<uint16_t *>(base)[32 + item] = (uint16_t)(blk[2] | (blk[3] << 8));
        } else if (item < 96) {  // scales of (g, sub-block): bytes (tile j/2, row g + 8*(j%2))
            const int g = (item - 32) / 8, s = (item - 32) % 8;
            uint32_t w = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint8_t *blk = q4k_block(j >> 1 ? wu : wg, H, e, I, jj * 16 + g + 8 * (j & 1), sb);
                w |= q4k_param(blk, s, 0) << (8 * j);
            }
            reinterpret_cast<uint32_t *>(base + kQ4kScaleOff)[g * 8 + s] = w;
        } else {  // mins of (lane, tile): A-fragment registers 0-1, k = sub-block
            const int lane = (item - 96) / 2, t = (item - 96) % 2;
            uint32_t w = 0;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint8_t *blk = q4k_block(t ? wu : wg, H, e, I, jj * 16 + frag_row(lane, r), sb);
#pragma unroll
                for (int h = 0; h < 2; ++h) w |= q4k_param(blk, frag_col(lane, r, h), 1) << (8 * (2 * r + h));
            }
            reinterpret_cast<uint32_t *>(base + kQ4kMinOff)[lane * 2 + t] = w;
        }
    }
}

}  // namespace spx

using namespace spx;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

extern "C" size_t spx_w4_packed_bytes(int E, int H, int I, int S) {
    if (E < 1 || H < 128 || I < 128 || (S != 16 && S != 32) || H % 128 || I % 128) return 0;
    return w4_colblk_offset(E, H, I, S) + w4_colblk_bytes(E, H, I);
}

extern "C" size_t spx_f16_packed_bytes(int E, int H, int I) {
    if (E < 1 || H < 128 || I < 16 || H % 128 || I % kF16S) return 0;
    return (size_t)E * (I / kF16S) * f16_unit_bytes(H);
}

extern "C" int spx_w4_repack(const int32_t *qw_gate, const uint16_t *s_gate, const int32_t *qw_up,
                             const uint16_t *s_up, const int32_t *qw_down, const uint16_t *s_down, int E, int H,
                             int I, int S, void *packed, spx_stream_t stream) {
    if (!qw_gate || !s_gate || !qw_up || !s_up || !qw_down || !s_down || !packed) return SPX_ERR_INVALID_ARG;
    if (E < 1 || H < 1 || I < 1) return SPX_ERR_INVALID_ARG;
    if ((S != 16 && S != 32) || H % 128 || I % 128 || H > kMaxH || E > kMaxE) return SPX_ERR_UNSUPPORTED;
    if (!aligned16(packed)) return SPX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(packed);
    const int spe = I / S;
    size_t tot = (size_t)E * spe * (H / 128) * 2 * S;
    w4_pack_scales<<<grid_for(tot), 256, 0, s>>>(s_gate, s_up, E, H, I, S, out);
    tot = (size_t)E * spe * ((H / 16) / (2 / (S / 16))) * 128;
    w4_pack_gu<<<grid_for(tot), 256, 0, s>>>(qw_gate, qw_up, E, H, I, S, out);
    tot = (size_t)E * spe * ((H / 16) / (4 / (S / 16))) * 128;
    w4_pack_down<<<grid_for(tot), 256, 0, s>>>(qw_down, E, H, I, S, out);
    int st = record_launch(cudaGetLastError());
    if (st) return st;
    cudaError_t e = cudaMemcpyAsync(out + w4_units_bytes(E, H, I, S), s_down, (size_t)E * (I / 128) * H * 2,
                                    cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return record_launch(e);
    uint8_t *cb = out + w4_colblk_offset(E, H, I, S);
    tot = (size_t)E * (H / 32) * (I / 128) * 32;
    w4_pack_colblk_scales<<<grid_for(tot), 256, 0, s>>>(s_down, E, H, I, cb);
    tot = (size_t)E * (H / 32) * (I / 128) * 512;
    w4_pack_colblk_codes<<<grid_for(tot), 256, 0, s>>>(qw_down, E, H, I, cb);
    return record_launch(cudaGetLastError());
}

// Q8_0 down once more in unit order for the expert launch: one thread per
// (unit, pair, lane, tile) writes the lane's 8 codes of that tile; then one
// thread per (expert, block of 32 intermediate rows, output) writes a scale.
__global__ void q8_pack_udn(const uint8_t *wd, int E, int H, int I, uint8_t *codes, uint16_t *scales) {
    const int spe = I / 16, NP = H / 32;
    const size_t total = (size_t)E * spe * NP * 32 * 2;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(idx & 1);
        const int lane = (int)((idx >> 1) & 31);
        const size_t up = idx >> 6;  // unit * NP + pair
        const int P = (int)(up % NP);
        const size_t unit = up / NP;
        const size_t e = unit / spe;
        const int j = (int)(unit % spe);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int jb = 0; jb < 8; ++jb) {
            const int r = jb >> 1;
            const int n = down_col(2 * P + q, frag_row(lane, r));
            const int k = j * 16 + frag_col(lane, r, jb & 1);
            w[jb >> 2] |= (uint32_t)q8_code(wd, I, e, H, n, k) << (8 * (jb & 3));
        }
        *reinterpret_cast<uint2 *>(codes + unit * ((size_t)H * 16) + (size_t)P * 512 + lane * 16 + q * 8) =
            make_uint2(w[0], w[1]);
    }
    const size_t ns = (size_t)E * (I / 32) * H;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < ns; idx += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(idx % H);
        const int b = (int)((idx / H) % (I / 32));
        const size_t e = idx / ((size_t)H * (I / 32));
        scales[idx] = q8_scale(wd, I, e, H, n, b);
    }
}

extern "C" size_t spx_gguf_packed_bytes(int E, int H, int I, int gate_up_type) {
    if (E < 1 || H < 128 || I < 128 || H % 128 || I % 128) return 0;
    if (gate_up_type == SPX_GGUF_Q8_0) return gguf_packed_total(E, H, I, kFmtQ8);
    if (gate_up_type == SPX_GGUF_Q2_K && H % 256 == 0) return gguf_packed_total(E, H, I, kFmtQ2K);
    if (gate_up_type == SPX_GGUF_Q4_K && H % 256 == 0) return gguf_packed_total(E, H, I, kFmtQ4K);
    return 0;
}

extern "C" int spx_gguf_repack(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down, int E, int H, int I,
                               int gate_up_type, void *packed, spx_stream_t stream) {
    if (!w_gate || !w_up || !w_down || !packed) return SPX_ERR_INVALID_ARG;
    if (E < 1 || H < 1 || I < 1) return SPX_ERR_INVALID_ARG;
    if (gate_up_type != SPX_GGUF_Q8_0 && gate_up_type != SPX_GGUF_Q2_K && gate_up_type != SPX_GGUF_Q4_K)
        return SPX_ERR_INVALID_ARG;
    if (H % 128 || I % 128 || H > kMaxH || E > kMaxE) return SPX_ERR_UNSUPPORTED;
    if (gate_up_type != SPX_GGUF_Q8_0 && H % 256) return SPX_ERR_UNSUPPORTED;
    if (!aligned16(packed)) return SPX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(packed);
    size_t units;
    if (gate_up_type == SPX_GGUF_Q8_0) {
        q8_pack_gu<<<grid_for((size_t)E * (I / 16) * (H / 128) * 512), 256, 0, s>>>(w_gate, w_up, E, H, I, out);
        units = q8_units_bytes(E, H, I);
    } else if (gate_up_type == SPX_GGUF_Q2_K) {
        q2k_pack_gu<<<grid_for((size_t)E * (I / 16) * (H / 256) * 512), 256, 0, s>>>(w_gate, w_up, E, H, I, out);
        units = q2k_units_bytes(E, H, I);
    } else {
        q4k_pack_gu<<<grid_for((size_t)E * (I / 16) * (H / 256) * 1024), 256, 0, s>>>(w_gate, w_up, E, H, I, out);
        units = q4k_units_bytes(E, H, I);
    }
    q8_pack_dn<<<grid_for((size_t)E * (H / 32) * (I / 128) * 512), 256, 0, s>>>(w_down, E, H, I, out + units);
    const int fmt = gate_up_type == SPX_GGUF_Q8_0 ? kFmtQ8 : gate_up_type == SPX_GGUF_Q2_K ? kFmtQ2K : kFmtQ4K;
    q8_pack_udn<<<grid_for((size_t)E * (I / 16) * (H / 32) * 64), 256, 0, s>>>(
        w_down, E, H, I, out + gguf_udn_offset(E, H, I, fmt),
        reinterpret_cast<uint16_t *>(out + gguf_uds_offset(E, H, I, fmt)));
    return record_launch(cudaGetLastError());
}

extern "C" size_t spx_w4_zeros_bytes(int E, int H, int I, int S) {
    if (!spx_w4_packed_bytes(E, H, I, S)) return 0;
    return w4_zeros_gu_bytes(E, H, I, S) + w4_zeros_dn_bytes(E, H, I);
}

extern "C" int spx_w4_zeros_repack(const int32_t *qz_gate, const int32_t *qz_up, const int32_t *qz_down, int E,
                                   int H, int I, int S, void *zeros, spx_stream_t stream) {
    if (!qz_gate || !qz_up || !qz_down || !zeros) return SPX_ERR_INVALID_ARG;
    if (E < 1 || H < 1 || I < 1) return SPX_ERR_INVALID_ARG;
    if ((S != 16 && S != 32) || H % 128 || I % 128 || H > kMaxH || E > kMaxE) return SPX_ERR_UNSUPPORTED;
    if (!aligned16(zeros)) return SPX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *out = static_cast<uint16_t *>(zeros);
    size_t tot = (size_t)E * (I / S) * (H / 128) * 2 * S;
    w4_pack_zeros_gu<<<grid_for(tot), 256, 0, s>>>(qz_gate, qz_up, E, H, I, S, out);
    tot = (size_t)E * (H / 32) * (I / 128) * 32;
    w4_pack_zeros_dn<<<grid_for(tot), 256, 0, s>>>(qz_down, E, H, I,
                                                   out + w4_zeros_gu_bytes(E, H, I, S) / sizeof(uint16_t));
    return record_launch(cudaGetLastError());
}

extern "C" size_t spx_shared_packed_bytes(int H, int I_s) {
    if (H < 128 || I_s < 16 || H % 128 || I_s % kF16S || H > kMaxH) return 0;
    return shared_packed_bytes(H, I_s);
}

extern "C" int spx_shared_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down, int H, int I_s,
                                 void *packed, spx_stream_t stream) {
    if (spx_shared_packed_bytes(H, I_s) == 0) return SPX_ERR_UNSUPPORTED;
    int st = spx_f16_repack(w_gate, w_up, w_down, 1, H, I_s, packed, stream);
    if (st) return st;
    const size_t tot = (size_t)(H / 32) * (I_s / 16) * 256;
    f16_pack_pairdown<<<grid_for(tot), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w_down, H, I_s, static_cast<uint8_t *>(packed) + shared_pairdown_offset(H, I_s));
    return record_launch(cudaGetLastError());
}

extern "C" int spx_f16_repack(const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down, int E, int H,
                              int I, void *packed, spx_stream_t stream) {
    if (!w_gate || !w_up || !w_down || !packed) return SPX_ERR_INVALID_ARG;
    if (E < 1 || H < 1 || I < 1) return SPX_ERR_INVALID_ARG;
    if (H % 128 || I % kF16S || H > kMaxH || E > kMaxE) return SPX_ERR_UNSUPPORTED;
    if (!aligned16(packed)) return SPX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(packed);
    const int spe = I / kF16S;
    size_t tot = (size_t)E * spe * (H / 16) * 2 * 128;
    f16_pack_gu<<<grid_for(tot), 256, 0, s>>>(w_gate, w_up, E, H, I, out);
    tot = (size_t)E * spe * (H / 32) * 2 * 128;
    f16_pack_down<<<grid_for(tot), 256, 0, s>>>(w_down, E, H, I, out);
    return record_launch(cudaGetLastError());
}
