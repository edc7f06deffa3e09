// spx_timeline.cuh -- phase marks of the draft launch, compiled only into the
// profiling build (libspx_timeline.so, -DSPX_TIMELINE); the product library
// has none of this code.
//
// Each launch writes into one of kTlSlots slots (the host passes the slot, so
// a chain of launches keeps every launch's marks apart); per block, kTlEvents
// 64-bit words.  "First" marks keep the smallest %globaltimer value (stored
// complemented under atomicMax, so a cleared word means "not set"), "last"
// marks the largest, sums add nanoseconds or counts.  The marks go to a
// shared-memory copy of the block's words (shared-memory atomics: no global
// memory operation is left in flight for a later fence to wait on) and the
// consumer warps copy them out once, at the end of the block.
#pragma once

#include <stdint.h>

namespace spx {

constexpr int kTlSlots = 8;
constexpr int kTlBlocks = 256;
constexpr int kTlEvents = 48;

enum TlEvent : int {
    TL_ENTRY = 0,          // first: block entered the kernel
    TL_PROD_STATIC = 1,    // first: producer issued its static unit's copies
    TL_PROD_GRIDDEP = 2,   // first: producer past griddepcontrol.wait
    TL_X_STAGED = 3,       // first: x (and its group sums) in shared memory
    TL_ROUTED = 4,         // first: routing published in shared memory
    TL_FIRST_FILL = 5,     // first: a consumer warp got its first stage fill
    TL_GU_LAST = 6,        // last: a gate/up item (shared or routed) finished
    TL_DN_W_FIRST = 7,     // first: a down item's weights landed
    TL_DN_H_FIRST = 8,     // first: a down item's intermediate landed
    TL_DN_LAST = 9,        // last: a down item finished
    TL_PROD_LAST = 10,     // last: producer issued its last item
    TL_CONS_DONE = 11,     // first: every consumer warp left the item loop
    TL_OUT_DONE = 12,      // last: output pass done (last block only)
    TL_SG_LAST = 13,       // last: shared gate/up item finished
    TL_RG_FIRST = 14,      // first: routed gate/up item started
    TL_RG_LAST = 15,       // last: routed gate/up item finished
    TL_W_FULL = 16,        // sum: consumer ns waiting for stage weights
    TL_W_HFULL = 17,       // sum: consumer ns waiting for a down item's intermediate
    TL_W_EMPTY = 18,       // sum: producer ns waiting for a free stage
    TL_N_SG = 19,          // sum: items of each kind
    TL_N_RG = 20,
    TL_N_SD = 21,
    TL_N_RD = 22,
    TL_EXIT = 23,          // last: a consumer thread left the kernel
    TL_RD_H_LAST = 24,     // last: a routed down item's intermediate landed
    TL_SD_LAST = 25,       // last: shared down item finished
    TL_W_POLL = 26,        // sum: ns from a down item's registration to its intermediate copy
    TL_BYTES = 27,         // sum: weight bytes the producer issued
    TL_W_TICKET = 28,      // sum: producer ns waiting for a queue ticket's value
    TL_N_TICKET = 29,      // sum: queue tickets used
    TL_W_ROUTE = 30,       // sum: producer ns waiting for the routing
    TL_ISSUE = 31,         // sum: producer ns inside a fill's issue (after the free stage)
    TL_P_SG = 32,          // sum: producer ns in shared gate/up units
    TL_P_RG = 33,          // sum: producer ns in routed gate/up units
    TL_P_DN = 34,          // sum: producer ns in down units
    TL_P_FENCE = 35,       // sum: producer ns in the down items' registration fence
    TL_P_SLOT = 36,        // sum: producer ns waiting for a gate/up slot
    TL_C_SG = 37,          // sum: consumer ns computing shared gate/up items (fill to release)
    TL_C_RG = 38,          // sum: ... routed gate/up items
    TL_C_SD = 39,          // sum: ... shared down items (intermediate landed to release)
    TL_C_RD = 40,          // sum: ... routed down items
    TL_C_GU_DONE = 41,     // sum: consumer ns completing gate/up blocks (slot sums, finalize, publish)
    TL_C_OUT = 42,         // sum: consumer ns adding down outputs to the accumulator
};

// Per-fill and per-item trace of two blocks (0 and gridDim/2) of each launch:
// times in ns after the block's entry, plain shared-memory stores (the
// producer is one thread; consumer items take a slot by a shared counter).
constexpr int kTrFills = 48, kTrItems = 64, kTrUnits = 16, kTrBlocks = 2;
struct TrBlock {
    uint32_t fill[kTrFills][4];  // wait start, stage free, issued, kind << 24 | bytes
    uint32_t item[kTrItems][4];  // warp << 8 | kind, fill landed, intermediate landed, done
    uint32_t unit[kTrUnits][4];  // start, queue unit, described, fills issued
    unsigned long long t0;
    uint32_t nitem, pad;
    uint32_t route[8];           // routing warp: start, selected, outputs, tables, published
};

}  // namespace spx

#if defined(SPX_TIMELINE) && defined(__CUDACC__)
namespace spx {
// one translation unit (the draft launch's) includes this header
__device__ unsigned long long g_tl[kTlSlots][kTlBlocks][kTlEvents];
__shared__ unsigned long long s_tl[kTlEvents];
__device__ TrBlock g_tr[kTlSlots][kTrBlocks];
__shared__ TrBlock s_tr;
__device__ __forceinline__ int tr_block() {
    return blockIdx.x == 0 ? 0 : (blockIdx.x == gridDim.x / 2 ? 1 : -1);
}
__device__ __forceinline__ uint32_t tr_now() { return (uint32_t)(global_timer_ns() - s_tr.t0); }
}  // namespace spx
// Per-block marks (a few per block): shared-memory atomics.  The per-fill and
// per-item marks are compiled out: their 64-bit shared atomics (compare-and-
// swap loops) slowed the very paths they measured; the trace covers them.
#define TLB_FIRST(slot, ev) atomicMax(&::spx::s_tl[(ev)], ~(unsigned long long)::spx::global_timer_ns())
#define TLB_LAST(slot, ev) atomicMax(&::spx::s_tl[(ev)], (unsigned long long)::spx::global_timer_ns())
#define TL_FIRST(slot, ev) ((void)0)
#define TL_LAST(slot, ev) ((void)0)
#define TL_ADD(slot, ev, v) ((void)0)
#define TL_NOW() ::spx::global_timer_ns()
#define TL_ON 1
// clear the block's shared words (before the block's first barrier)
#define TL_INIT()                                                                                   \
    do {                                                                                            \
        for (int i_ = threadIdx.x; i_ < ::spx::kTlEvents; i_ += blockDim.x) ::spx::s_tl[i_] = 0;    \
        uint32_t *w_ = reinterpret_cast<uint32_t *>(&::spx::s_tr);                                   \
        for (int i_ = threadIdx.x; i_ < (int)(sizeof(::spx::TrBlock) / 4); i_ += blockDim.x) w_[i_] = 0; \
        if (threadIdx.x == 0) ::spx::s_tr.t0 = ::spx::global_timer_ns();                             \
    } while (0)
// copy the block's words out (consumer threads ctid, after the block's last barrier)
#define TL_FLUSH(slot, ctid)                                                                          \
    do {                                                                                               \
        if ((ctid) < ::spx::kTlEvents && blockIdx.x < ::spx::kTlBlocks)                               \
            ::spx::g_tl[(slot) & (::spx::kTlSlots - 1)][blockIdx.x][(ctid)] = ::spx::s_tl[(ctid)];    \
        const int tb_ = ::spx::tr_block();                                                            \
        if (tb_ >= 0) {                                                                               \
            const uint32_t *src_ = reinterpret_cast<const uint32_t *>(&::spx::s_tr);                  \
            uint32_t *dst_ = reinterpret_cast<uint32_t *>(&::spx::g_tr[(slot) & (::spx::kTlSlots - 1)][tb_]); \
            for (int i_ = (ctid); i_ < (int)(sizeof(::spx::TrBlock) / 4); i_ += 32 * 11) dst_[i_] = src_[i_]; \
        }                                                                                             \
    } while (0)
#define TR_ON() (::spx::tr_block() >= 0)
#define TR_NOW() ::spx::tr_now()
// waits for v (a queue ticket in flight) by storing it to a shared word, and
// counts the wait
#define TL_TICKET(slot, v, sinkp) ((void)0)
#else
#define TLB_FIRST(slot, ev) ((void)0)
#define TLB_LAST(slot, ev) ((void)0)
#define TL_FIRST(slot, ev) ((void)0)
#define TL_LAST(slot, ev) ((void)0)
#define TL_ADD(slot, ev, v) ((void)0)
#define TL_NOW() 0ull
#define TL_ON 0
#define TL_INIT() ((void)0)
#define TL_FLUSH(slot, ctid) ((void)0)
#define TR_ON() false
#define TR_NOW() 0u
#define TL_TICKET(slot, v, sinkp) ((void)0)
#endif
