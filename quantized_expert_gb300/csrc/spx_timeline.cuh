// spx_timeline.cuh -- phase marks of the draft launch, compiled only into the
// profiling build (libspx_timeline.so, -DSPX_TIMELINE); the product library
// has none of this code.
//
// Each launch writes into one of kTlSlots slots (the host passes the slot, so
// a chain of launches keeps every launch's marks apart); per block, kTlEvents
// 64-bit words.  "First" marks keep the smallest %globaltimer value (stored
// complemented under atomicMax, so a cleared word means "not set"), "last"
// marks the largest, sums add nanoseconds or counts.
#pragma once

#include <stdint.h>

namespace spx {

constexpr int kTlSlots = 8;
constexpr int kTlBlocks = 256;
constexpr int kTlEvents = 32;

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
};

}  // namespace spx

#if defined(SPX_TIMELINE) && defined(__CUDACC__)
namespace spx {
// one translation unit (the draft launch's) includes this header
__device__ unsigned long long g_tl[kTlSlots][kTlBlocks][kTlEvents];
__device__ __forceinline__ unsigned long long *tl_word(int slot, int ev) {
    return &g_tl[slot & (kTlSlots - 1)][blockIdx.x < kTlBlocks ? blockIdx.x : kTlBlocks - 1][ev];
}
}  // namespace spx
#define TL_FIRST(slot, ev) atomicMax(::spx::tl_word((slot), (ev)), ~(unsigned long long)::spx::global_timer_ns())
#define TL_LAST(slot, ev) atomicMax(::spx::tl_word((slot), (ev)), (unsigned long long)::spx::global_timer_ns())
#define TL_ADD(slot, ev, v) atomicAdd(::spx::tl_word((slot), (ev)), (unsigned long long)(v))
#define TL_NOW() ::spx::global_timer_ns()
#define TL_ON 1
// waits for v (a queue ticket in flight) by storing it to a shared word, and
// counts the wait
#define TL_TICKET(slot, v, sinkp)                                     \
    do {                                                              \
        const unsigned long long t_ = TL_NOW();                       \
        *(volatile uint32_t *)(sinkp) = (v);                          \
        TL_ADD((slot), ::spx::TL_W_TICKET, TL_NOW() - t_);            \
        TL_ADD((slot), ::spx::TL_N_TICKET, 1);                        \
    } while (0)
#else
#define TL_FIRST(slot, ev) ((void)0)
#define TL_LAST(slot, ev) ((void)0)
#define TL_ADD(slot, ev, v) ((void)0)
#define TL_NOW() 0ull
#define TL_ON 0
#define TL_TICKET(slot, v, sinkp) ((void)0)
#endif
