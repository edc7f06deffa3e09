// spx_internal.cuh -- shared device helpers and packed-format geometry for libspx.
// sm_103a only: inline PTX for mbarriers, bulk copies (TMA engine), the
// m16n8k16 tensor-core instruction and LOP3; nothing here is portable on purpose.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/spx.h"

namespace spx {

// ---------------------------------------------------------------- limits --
constexpr int kMaxT = 64;          // tokens per call
constexpr int kMaxE = 256;         // experts
constexpr int kMaxSlots = 512;     // T * k
constexpr int kMaxH = 8192;
constexpr int kGroup = 128;        // GPTQ group size along K
constexpr int kChunk = 16384;      // bytes per ring stage
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kSmemLimit = 227 * 1024;

// --------------------------------------------------------- workspace ---
// Header of the caller's workspace (zeroed once; kernels leave it zeroed).
struct WsHeader {
    uint32_t work_counter;   // dynamic unit queue of the expert launch
    uint32_t done_ticket;    // completed blocks of the expert launch
    int32_t status;          // SPX_OK or SPX_ERR_TIMEOUT (sticky)
    uint32_t route_ticket;   // completed blocks of the router product
    uint32_t exit_ticket;    // blocks of the expert launch done with its output pass
    int32_t timeout_site;    // which bounded wait gave up first (with status; 0 = none)
    uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");
static_assert(offsetof(WsHeader, timeout_site) - offsetof(WsHeader, status) == 3 * sizeof(int32_t),
              "a wait that holds &status records its site three words on");
// Bounded waits that give up record their site next to the status word.
enum : int32_t { SITE_ALL_SYNC = 1, SITE_FILL = 2, SITE_HSLICE = 3, SITE_GATE = 4, SITE_ROUTING = 5, SITE_SLOT = 6,
                 SITE_STAGE = 7, SITE_POLLER = 8, SITE_ENGINE = 9, SITE_TC = 10 };
#if defined(__CUDACC__)
__device__ __forceinline__ void record_timeout(int32_t *status, int32_t site) {
    atomicCAS(status, 0, (int32_t)SPX_ERR_TIMEOUT);
    atomicCAS(status + 3, 0, site);
}
#endif
constexpr size_t kWsAccOffset = 256;


// ----------------------------------------------------- packed geometry ---
// INT4 unit (S = 16*MS columns of I):
//   [gate/up: H/128 groups; group = 2S fp16 scales (gate cols, then up cols)
//             followed by the group's 8 k-steps of codes as 512 B blocks of
//             KB = 2/MS k-steps (32 lanes x 16 B; a lane's 4 words = [ks][tile])]
//   [down   : (H/16)/MB blocks of 512 B, MB = 4/MS m-tiles per block
//             (a lane's 4 words = [tile][ks])]
// then after all units: down scales [E][I/128][H] fp16 (canonical).
__host__ __device__ inline size_t w4_group_bytes(int S) { return (size_t)132 * S; }
__host__ __device__ inline size_t w4_gu_bytes(int H, int S) { return (size_t)(H / 128) * w4_group_bytes(S); }
__host__ __device__ inline size_t w4_dn_bytes(int H, int S) { return (size_t)H * S / 2; }
__host__ __device__ inline size_t w4_unit_bytes(int H, int S) { return w4_gu_bytes(H, S) + w4_dn_bytes(H, S); }
__host__ __device__ inline size_t w4_units_bytes(int E, int H, int I, int S) {
    return (size_t)E * (I / S) * w4_unit_bytes(H, S);
}
// INT4 down weights again, column-block-major (for the split-K draft launch):
// per expert, per pair of output m-tiles (32 columns), per group of 128 rows
// of I: 32 fp16 scales in tile-row order (tile q row m at q*16 + m) followed
// by 4 blocks of 512 B, each 2 k-steps: lane words [ks][tile].
constexpr int kW4ColGroupBytes = 64 + 4 * 512;
__host__ __device__ inline size_t w4_colblk_bytes(int E, int H, int I) {
    return (size_t)E * (H / 32) * (I / 128) * kW4ColGroupBytes;
}
// Zero points of asymmetric INT4 experts (a buffer of their own): gate/up
// [E][I/S][H/128][2S] fp16, then down [E][H/32][I/128][32] fp16.
__host__ __device__ inline size_t w4_zeros_gu_bytes(int E, int H, int I, int S) {
    return (size_t)E * (I / S) * (H / 128) * 2 * S * 2;
}
__host__ __device__ inline size_t w4_zeros_dn_bytes(int E, int H, int I) {
    return (size_t)E * (H / 32) * (I / 128) * 32 * 2;
}
constexpr int kFmtQ8 = 2;   // EngineParams::routed_fmt of GGUF Q8_0 experts
constexpr int kFmtQ2K = 3;  // ... of GGUF Q2_K gate/up with Q8_0 down
constexpr int kFmtQ4K = 4;  // ... of GGUF Q4_K gate/up with Q8_0 down
constexpr int kFmtW4Z = 5;  // expert-launch instance of INT4 with zero points (routed_fmt stays 0)
// GGUF Q8_0 experts (draft launch only; S = 16).  A group of 128 rows is four
// Q8_0 blocks of 32 rows: 4 x 32 fp16 scales ([block][tile-row order], as the
// INT4 scales) followed by the group's 8 k-steps of codes, 512 B each (32
// lanes x 16 B; a lane's 16 B = tile 0's 8 codes, then tile 1's; code byte j
// of a tile is register j/2, half j%2 of its A fragment).
//   gate/up units [E][I/16]: H/128 groups (tiles: gate, up);
//   then down, column-block-major [E][H/32][I/128] groups (tiles: the pair's two).
constexpr int kQ8ScaleBytes = 4 * 32 * 2;
constexpr int kQ8GroupBytes = kQ8ScaleBytes + 8 * 512;
__host__ __device__ inline size_t q8_unit_bytes(int H) { return (size_t)(H / 128) * kQ8GroupBytes; }
__host__ __device__ inline size_t q8_units_bytes(int E, int H, int I) { return (size_t)E * (I / 16) * q8_unit_bytes(H); }
__host__ __device__ inline size_t q8_packed_bytes(int E, int H, int I) {
    return q8_units_bytes(E, H, I) + (size_t)E * (H / 32) * (I / 128) * kQ8GroupBytes;
}
// GGUF Q2_K gate/up (draft launch only; S = 16; H a multiple of 256), one
// super-block of 256 rows of a slice's two tiles (gate, up) in 2688 bytes:
//   d [32] fp16, dmin [32] fp16 (tile-row order t*16 + m);
//   sub-block scales [g 0..7][k-step 0..15] u16, nibble j = (tile j/2, row
//     g + 8*(j%2)) at bits 4j;
//   mins [lane][tile] u32 in A-fragment order (k = sub-block): nibble of
//     register r, half h at bits 16h + 4r;
//   codes: 4 blocks of 512 B, each 4 k-steps (32 lanes x 16 B; lane word =
//     one k-step, code of tile t, register r, half h at bits 16h + 2(4t + r)).
// Gate/up units [E][I/16] of H/256 super-blocks, then the down projection in
// the Q8_0 column-block-major layout.
constexpr int kQ2kScaleOff = 128;
constexpr int kQ2kMinOff = kQ2kScaleOff + 8 * 16 * 2;
constexpr int kQ2kCodeOff = kQ2kMinOff + 32 * 2 * 4;
constexpr int kQ2kSbBytes = kQ2kCodeOff + 4 * 512;
static_assert(kQ2kSbBytes == 2688, "Q2_K super-block of a slice: 2.625 bits per weight");
__host__ __device__ inline size_t q2k_unit_bytes(int H) { return (size_t)(H / 256) * kQ2kSbBytes; }
__host__ __device__ inline size_t q2k_units_bytes(int E, int H, int I) {
    return (size_t)E * (I / 16) * q2k_unit_bytes(H);
}
// GGUF Q4_K gate/up (draft launch only; S = 16; H a multiple of 256), one
// super-block of 256 rows of a slice's two tiles in 4736 bytes:
//   d [32] fp16, dmin [32] fp16 (tile-row order t*16 + m);
//   sub-block scales [g 0..7][sub-block 0..7] u32, byte j = (tile j/2, row
//     g + 8*(j%2)), 6-bit values;
//   mins [lane][tile] u32: bytes (row g, sub-block 2c), (g, 2c+1), (g+8, 2c),
//     (g+8, 2c+1) with c = lane%4 (the A fragment's registers 0-1, k = sub-block);
//   codes: 8 blocks of 512 B, each 2 k-steps (32 lanes x 16 B; lane words
//     [k-step][tile], code of register r, half h at bits 16h + 4r).
constexpr int kQ4kScaleOff = 128;
constexpr int kQ4kMinOff = kQ4kScaleOff + 8 * 8 * 4;
constexpr int kQ4kCodeOff = kQ4kMinOff + 32 * 2 * 4;
constexpr int kQ4kSbBytes = kQ4kCodeOff + 8 * 512;
static_assert(kQ4kSbBytes == 4736, "Q4_K super-block of a slice: 4.625 bits per weight");
__host__ __device__ inline size_t q4k_unit_bytes(int H) { return (size_t)(H / 256) * kQ4kSbBytes; }
__host__ __device__ inline size_t q4k_units_bytes(int E, int H, int I) {
    return (size_t)E * (I / 16) * q4k_unit_bytes(H);
}
// GGUF experts for the expert launch (draft calls above 5 tokens and
// cache-aware ones): after the draft launch's layout, the Q8_0 down codes
// again in unit order [E][I/16], a unit = H/32 blocks of 512 B, one per m-tile
// pair P (32 lanes x 16 B: tile 0's 8 codes, then tile 1's, A[m][kc] = code of
// W_down[down_col(2P+q, m)][16 j + kc]), then the down scales [E][I/32][H] fp16.
__host__ __device__ inline size_t gguf_gu_units_bytes(int E, int H, int I, int fmt) {
    return fmt == kFmtQ8 ? q8_units_bytes(E, H, I) : fmt == kFmtQ2K ? q2k_units_bytes(E, H, I) : q4k_units_bytes(E, H, I);
}
__host__ __device__ inline size_t gguf_udn_offset(int E, int H, int I, int fmt) {
    return gguf_gu_units_bytes(E, H, I, fmt) + (q8_packed_bytes(E, H, I) - q8_units_bytes(E, H, I));
}
__host__ __device__ inline size_t gguf_uds_offset(int E, int H, int I, int fmt) {
    return gguf_udn_offset(E, H, I, fmt) + (size_t)E * (I / 16) * H * 16;
}
__host__ __device__ inline size_t gguf_packed_total(int E, int H, int I, int fmt) {
    return gguf_uds_offset(E, H, I, fmt) + (size_t)E * (I / 32) * H * 2;
}
__host__ __device__ inline size_t w4_colblk_offset(int E, int H, int I, int S) {
    return w4_units_bytes(E, H, I, S) + (size_t)E * (I / 128) * H * 2;
}
// FP16 unit (S = 16):
//   [gu  : H/16 blocks (one k-step each) of 2 tiles x 32 lanes x 16 B]
//   [down: H/32 blocks (one m-tile pair each) of 2 tiles x 32 lanes x 16 B]
constexpr int kF16S = 16;
__host__ __device__ inline size_t f16_unit_bytes(int H) { return (size_t)6 * H * kF16S; }
__host__ __device__ inline size_t f16_gu_bytes(int H) { return (size_t)4 * H * kF16S; }
// Shared expert pack = FP16 units (one expert) followed by its down weights in
// pair-major order: per m-tile pair P, per k-step of I: [tile][lane] x 16 B.
__host__ __device__ inline size_t shared_pairdown_offset(int H, int I) { return (size_t)(I / kF16S) * f16_unit_bytes(H); }
__host__ __device__ inline size_t shared_packed_bytes(int H, int I) {
    return shared_pairdown_offset(H, I) + (size_t)(H / 32) * (I / 16) * 1024;
}

// Per-expert token table (workspace), written by the routing launch or by the
// table launch of the unit calls, bulk-copied next to the expert's first chunk.
struct TokEntry {
    int32_t tok;    // row of x
    int32_t row;    // output row (token, or sorted position)
    float scale;    // output scale (gate weight, or 1)
    int32_t pad;
};
struct TokTable {
    int32_t n;
    int32_t pad[3];
    TokEntry e[kMaxT];
};
constexpr size_t kTableBytes = sizeof(TokTable);  // 16 + 64*16
static_assert(kTableBytes % 16 == 0, "table is bulk-copied");
__host__ __device__ inline size_t ws_tables_offset(int T, int H) {
    return kWsAccOffset + ((size_t)T * H * 4 + 255) / 256 * 256;
}
// After the token tables: the expert launch's queue order of the active
// experts (kMaxE ints; cache-aware calls).
__host__ __device__ inline size_t ws_order_offset(int T, int H) {
    return ws_tables_offset(T, H) + (size_t)kMaxE * kTableBytes;
}

// Physical output column of row m (0..15) of down tile mt: tile pair P = mt/2
// covers 32 columns; rows (g, g+8) of tile q land on columns 4g+2q, 4g+2q+1,
// so one lane's C fragments of a pair are 4 consecutive columns of a token.
__host__ __device__ inline int down_col(int mt, int m) {
    return 32 * (mt >> 1) + 4 * (m & 7) + 2 * (mt & 1) + (m >> 3);
}
// Row/column of an m16k16 A-fragment element: lane (g = lane/4, c = lane%4),
// register r (0..3), half h (0..1).
__host__ __device__ inline int frag_row(int lane, int r) { return (lane >> 2) + 8 * (r & 1); }
__host__ __device__ inline int frag_col(int lane, int r, int h) { return 2 * (lane & 3) + h + 8 * (r >> 1); }

#if defined(__CUDACC__)
// ------------------------------------------------------------- PTX ------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: gives up after `budget_ns` of wall time (or at once when
// *abort is already set), records SPX_ERR_TIMEOUT in the status word and
// sets *abort so every later wait in the block returns immediately.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  int32_t *status, uint64_t budget_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > budget_ns) {
            record_timeout(status, SITE_ALL_SYNC);
            *abort = 1;
            return false;
        }
    }
}
// Bulk copy (TMA engine, no tensor map): global -> shared, completion counted
// on an mbarrier in bytes.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// 16-byte asynchronous global -> shared copy (completion: cp_async_wait_all
// of the issuing thread).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Bulk copy without an L2 hint (data that other blocks read as well).
__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ uint2 lds64(const void *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ uint32_t lds32(const void *p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}
// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// One packed INT4 word -> one m16k16 A fragment (4 x half2) holding code-8.
// OR-ing a nibble into the mantissa of fp16 1024.0 (0x6400) gives 1024 + q
// exactly; subtracting 1032 leaves q - 8.  The nibble in bits 4..7 of each
// half gives 1024 + 16q; a fused (x/16 - 72) gives q - 8.  Nibble j of the word
// is register (j & 3), half (j >> 2).
__device__ __forceinline__ void dequant_frag(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t kMagic = 0x64006400u, kLo = 0x000F000Fu, kHi = 0x00F000F0u;
    const uint32_t w8 = w >> 8;
    const __half2 sub = u32_as_h2(0x64086408u);   // (1032, 1032)
    const __half2 mul = u32_as_h2(0x2C002C00u);   // (1/16, 1/16)
    const __half2 add = u32_as_h2(0xD480D480u);   // (-72, -72)
    a[0] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w, kLo, kMagic)), sub));
    a[1] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, kHi, kMagic)), mul, add));
    a[2] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w8, kLo, kMagic)), sub));
    a[3] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w8, kHi, kMagic)), mul, add));
}
// Eight Q8_0 codes (w0: registers 0-1, w1: registers 2-3) -> one m16k16 A
// fragment of exact fp16 codes.  Flipping the sign bit makes the byte
// code + 128; placed under fp16 1024.0's exponent it gives 1152 + code, and
// subtracting 1152 leaves the code (|code| <= 128, exact).
__device__ __forceinline__ void q8_frag(uint32_t w0, uint32_t w1, uint32_t (&a)[4]) {
    const uint32_t kExp = 0x64646464u;
    const __half2 sub = u32_as_h2(0x64806480u);  // (1152, 1152)
    const uint32_t f0 = w0 ^ 0x80808080u, f1 = w1 ^ 0x80808080u;
    a[0] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(f0, kExp, 0x4140)), sub));
    a[1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(f0, kExp, 0x4342)), sub));
    a[2] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(f1, kExp, 0x4140)), sub));
    a[3] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(f1, kExp, 0x4342)), sub));
}
// One packed INT4 word -> the same fragment positions holding the raw
// magic-exponent values: registers 0 and 2 (rows m < 8) get 1024 + q,
// registers 1 and 3 (rows m >= 8) get 1024 + 16 q, all exact in fp16.  The
// caller removes the 1024 (+8 zero point) and the factor 16 after the mma.
__device__ __forceinline__ void codes_frag(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t kMagic = 0x64006400u, kLo = 0x000F000Fu, kHi = 0x00F000F0u;
    const uint32_t w8 = w >> 8;
    a[0] = lop3_and_or(w, kLo, kMagic);
    a[1] = lop3_and_or(w, kHi, kMagic);
    a[2] = lop3_and_or(w8, kLo, kMagic);
    a[3] = lop3_and_or(w8, kHi, kMagic);
}
#endif  // __CUDACC__


// ------------------------------------------------------- launch params --
struct RouteParams {
    const __half *x;
    const __half *w_router;  // nullable: logits are given
    float *logits;
    int T, H, E, k, renorm;
    int32_t *topk_ids;
    float *topk_w;
    uint32_t *elb;  // nullable
    int layer;
    int32_t *counts, *offsets, *sorted_slots, *active, *n_active;  // all or none
    TokTable *tables;  // nullable: per-expert token tables (row = token, scale = weight)
    const uint8_t *resident;  // nullable (with order): resident experts are queued first
    int32_t *order;           // nullable: queue order of the active experts (expert launch)
    WsHeader *hdr;
};

struct EngineParams {
    // routed experts (packed units)
    const uint8_t *routed;
    const __half *w4_sdown;  // INT4: down scales [E][I/128][H]
    const uint8_t *w4_zeros; // INT4, nullable: repacked per-group zero points (else 8)
    int routed_fmt;          // 0 INT4, 1 FP16, kFmtQ8 / kFmtQ2K / kFmtQ4K GGUF (draft launch only)
    int S;                   // routed slice width (INT4: 16/32; FP16: 16)
    int E, I, k;
    int routed_enabled;
    const int32_t *active, *n_active;
    const int32_t *order;    // nullable: queue order of the active experts (else active)
    const uint32_t *ready;   // nullable: wait for ready[e] != 0 before streaming expert e
    const TokTable *tables;  // per expert, in the workspace
    // shared expert (FP16, S = 16), nullable
    const uint8_t *shared;
    const __half *w_sgate;
    int I_s;
    // problem
    const __half *x;
    int T, H;
    // output
    int mode;      // 0 sorted rows, 1 accumulate (gamma-scaled), 2 layer (weighted, last block writes out)
    float *yout;   // mode 0: y_sorted; otherwise the fp32 accumulator
    __half *out;   // mode 2: final fp16 output
    WsHeader *hdr;
    // geometry (set by the launcher)
    int groups;    // consumer warp groups (1 or 2)
    int nstages;   // ring stages per group
    int chunk;     // weight bytes per stage
    int npad;      // token columns of the shared scratch: 8 * ceil(T / 8)
    uint64_t wait_budget_ns;
};

int launch_route(const RouteParams &p, cudaStream_t s, bool pdl);
int route_validate(const uint16_t *x, const uint16_t *w_router, const float *logits, int T, int H, int E, int k,
                   const int32_t *ids, const float *w);
int launch_engine(const EngineParams &p, cudaStream_t s, bool pdl);
int engine_fits(int T, int H, int fmt, int S);
int engine_nt(int T);
// Routing done inside the draft launch (layer call): every block selects the
// experts of the T tokens from the logits itself; block 0 writes the outputs.
struct DraftRouting {
    const float *logits;  // [T][E]
    int renorm;
    int32_t *topk_ids;
    float *topk_w;
    uint32_t *elb;        // nullable
    int layer;
    int32_t *counts, *offsets, *sorted_slots, *active, *n_active;
};
// kq: GGUF K-quant gate/up (Q2_K, Q4_K): H a multiple of 256, S = 16, room for x sums
// Calls of at most this many tokens take the draft launch.  Its token loop would
// take up to 8 (one n-tile), but from 6 tokens on the routing launch + expert
// launch is as fast or faster (measured on GB300 at 5-8 tokens on the DeepSeek-,
// Qwen- and Phi-shaped layers), so larger calls go there.
constexpr int kDraftLaunchMaxT = 5;
bool draft_supported(int T, int H, int I, int S, int I_s, int E = 1, int k = 1, bool kq = false);
size_t draft_scratch_end(size_t base, int T, int H, int I, int I_s, int nact_max);
// rt == nullptr: routing from e.active / e.n_active and the token tables e.tables.
int launch_draft(const EngineParams &e, const DraftRouting *rt, size_t ws_scratch_base, bool pdl, cudaStream_t s);
int launch_router_logits(const __half *x, const __half *wr, int T, int H, int E, float *logits, cudaStream_t s,
                         bool pdl);
int launch_tables(const int32_t *offsets, const int32_t *sorted_slots, const int32_t *active,
                  const int32_t *n_active, int T, int k, int E, TokTable *tables, cudaStream_t s);

// Verify experts on the tensor-memory launches (spx_tc.cu): FP16 experts in
// that path's tile pack, a routing launch's token tables, the layer's fp32
// accumulator.
struct TcArgs {
    const __half *x;
    int T, H, E, I, k, I_s;
    const void *routed_tc;                                        // spx_f16_tc_repack pack of the routed experts
    const void *shared_tc;                                        // the shared expert's, or null
    const __half *w_sgate;                                        // nullable
    const int32_t *active, *n_active;
    const TokTable *tables;
    void *scratch;  // tc_scratch_bytes(), 1024-byte aligned
    float *acc;     // [T][H], zero on entry and on exit
    __half *out;
    WsHeader *hdr;
    uint64_t wait_budget_ns;
};
// Verify calls of at least kTcMinT tokens take the tensor-memory launches
// when the experts' tile packs are given.  Measured on GB300 (DeepSeek-, Qwen-
// and Phi-shaped layers, µs per layer, expert launch -> tensor-memory
// launches): 9 tokens 88.9 -> 86.8, 104.7 -> 103.8, 263.2 -> 244.1; 17 tokens
// 127.0 -> 114.4, 152.8 -> 140.9, 424.8 -> 313.0; from 33 tokens the expert
// launch is 40% slower or has no geometry (its activation rows stay in shared
// memory; the tensor-memory launches stream them).
constexpr int kTcMinT = 9;
inline bool tc_preferred(int T) { return T >= kTcMinT; }
// Workspace bytes of a call: launch 0 = spx_workspace_size (room for whichever
// launches the automatic choice may take), 1 = without the tensor-memory
// launches' scratch, 2 = spx_workspace_size_tc.
size_t workspace_bytes(int T, int H, int I, int E, int k, int I_s, int launch);
size_t tc_scratch_bytes(int T, int H, int I, int E, int k, int I_s);
size_t tc_tiles(int H, int I);  // 16 KB tiles of one expert's pack
int launch_tc_repack(const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int E, int H, int I, void *dst,
                     cudaStream_t s);
// The launches' parameters (tensor maps encoded, every pointer checked): made
// before anything of the call is enqueued, launched after the routing launch.
struct alignas(128) TcPlan {
    unsigned char bytes[2048];
};
int tc_plan(const TcArgs &a, TcPlan *plan);
int launch_tc_plan(const TcPlan &plan, cudaStream_t s, bool pdl);
int tc_preload();

// -------------------------------------------------------- host helpers --
int device_sm_count();
int record_launch(cudaError_t e);
// Load every kernel the layer call can launch on the current device (and set
// its shared-memory limit), so that later launches load no code.
int route_preload();
int engine_preload();
int draft_preload();
// The layer call: validates every argument, then (clear != nullptr) zeroes
// clear_bytes of `clear` on the stream, then enqueues the launches.
int moe_layer(const spx_layer_args *a, cudaStream_t s, void *clear, size_t clear_bytes);

}  // namespace spx
