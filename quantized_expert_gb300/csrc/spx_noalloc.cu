// spx_noalloc.cu -- the composite layer call for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc at the point where they
// run a layer: code that runs inside a custom allocator or a memory-pool
// callback, embedded runtimes that forbid device allocation after start-up,
// or hosts that must never block on the allocator's device-wide
// synchronisation.  They cannot provide the workspace that spx_moe_layer asks
// for.  spx_moe_layer_noalloc runs the same layer with its scratch (queue
// counter, completion ticket, status word, fp32 accumulator, token tables) in
// a fixed array that is part of the library image on every GPU that loads it.
#include "spx_internal.cuh"

#include <mutex>

namespace spx {

// Scratch of spx_moe_layer_noalloc: 1 MiB, held by every GPU that loads the
// library until the process exits.  Enough for any layer whose
// spx_workspace_size(T, H, I, E, k, I_s) is at most 1 MiB (for example the
// DeepSeek-V2-Lite-shaped layer at T = 1 and at T = 17).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mutex;
static void *g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in for the symbol and must never be
// passed to a kernel; the address comes from cudaGetSymbolAddress, looked up
// once per device with that device current.
static int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return record_launch(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPX_OK;
}

}  // namespace spx

using namespace spx;

extern "C" int spx_moe_layer_noalloc(const spx_layer_args *args, spx_stream_t stream) {
    if (!args) return SPX_ERR_INVALID_ARG;
    const int I = args->mode != 0 ? (args->f16 ? args->f16->I : 0)
                                  : args->gguf ? args->gguf->I : (args->w4 ? args->w4->I : 0);
    const int I_s = args->shared ? args->shared->I_s : 0;
    const size_t need = spx_workspace_size(args->T, args->H, I, args->E, args->k, I_s);
    if (need == 0) return SPX_ERR_UNSUPPORTED;
    if (need > kNoAllocScratchBytes) return SPX_ERR_WORKSPACE;  // T*H beyond the fixed scratch
    void *scratch = nullptr;
    int st = noalloc_scratch(&scratch);
    if (st) return st;
    // The array keeps the previous call's contents: clear the part this shape
    // uses (counters, tickets, status, accumulators), which must start at zero.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = cudaMemsetAsync(scratch, 0, need, s);
    if (e != cudaSuccess) return record_launch(e);
    spx_layer_args a = *args;
    a.ws = scratch;
    a.ws_bytes = kNoAllocScratchBytes;
    return spx_moe_layer(&a, stream);
}
