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
//
// Loading the library's code onto a device is itself an allocation (with lazy
// module loading, the default, it happens at the first use of a kernel or a
// device symbol), so it is done by spx_noalloc_init at start-up, once per
// device; the layer call refuses a device that was not set up.
#include "spx_internal.cuh"

#include <mutex>

namespace spx {

// Scratch of spx_moe_layer_noalloc: 1 MiB, held by every GPU that loads the
// library until the process exits.  Enough for any layer whose workspace
// without the tensor-memory verify launches' scratch is at most 1 MiB (for
// example the DeepSeek-V2-Lite-shaped layer at T = 1 and at T = 17); a verify
// call whose automatic choice would take those launches takes the expert
// launch here when their scratch does not fit.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mutex;
static bool g_noalloc_ready[64] = {};

static int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= 64) return SPX_ERR_CUDA;
    return SPX_OK;
}

// Device address of the scratch array on the current device (set up by
// spx_noalloc_init).  The host-side name g_noalloc_scratch is only a stand-in
// for the symbol and must never be passed to a kernel; the address comes from
// cudaGetSymbolAddress with the device current.  It is looked up on every
// call (a host-side table lookup once the module is loaded), so no address
// outlives the context it belongs to.
static int noalloc_scratch(void **out) {
    int dev = 0;
    int st = current_device(&dev);
    if (st) return st;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_ready[dev]) return SPX_ERR_WORKSPACE;  // spx_noalloc_init was not called here
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return record_launch(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    *out = p;
    return SPX_OK;
}

}  // namespace spx

using namespace spx;

extern "C" int spx_noalloc_init(void) {
    int dev = 0;
    int st = current_device(&dev);
    if (st) return st;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ready[dev]) return SPX_OK;
    // every kernel the layer call can launch, and the scratch symbol
    st = route_preload();
    if (!st) st = engine_preload();
    if (!st) st = draft_preload();
    if (!st) st = tc_preload();
    if (st) return st;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return record_launch(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_noalloc_ready[dev] = true;
    return SPX_OK;
}

extern "C" int spx_moe_layer_noalloc(const spx_layer_args *args, spx_stream_t stream) {
    if (!args) return SPX_ERR_INVALID_ARG;
    const int I = args->mode != 0 ? (args->f16 ? args->f16->I : 0)
                                  : args->gguf ? args->gguf->I : (args->w4 ? args->w4->I : 0);
    const int I_s = args->shared ? args->shared->I_s : 0;
    spx_layer_args a = *args;
    const int launch = args->mode == 1 ? args->verify_launch : 1;
    size_t need = workspace_bytes(args->T, args->H, I, args->E, args->k, I_s, launch);
    if (launch == 0 && need > kNoAllocScratchBytes) {
        // the tensor-memory verify launches' scratch does not fit: the expert launch serves the call
        a.verify_launch = 1;
        need = workspace_bytes(args->T, args->H, I, args->E, args->k, I_s, 1);
    }
    if (need == 0) return SPX_ERR_UNSUPPORTED;
    if (need > kNoAllocScratchBytes) return SPX_ERR_WORKSPACE;  // T*H beyond the fixed scratch
    void *scratch = nullptr;
    int st = noalloc_scratch(&scratch);
    if (st) return st;
    a.ws = scratch;
    a.ws_bytes = kNoAllocScratchBytes;
    // The array keeps the previous call's contents: the layer call clears the
    // part this shape uses (counters, tickets, status, accumulators), which
    // must start at zero, once every argument has been checked.
    return moe_layer(&a, reinterpret_cast<cudaStream_t>(stream), scratch, need);
}

extern "C" int spx_noalloc_status(int32_t *status, spx_stream_t stream) {
    if (!status) return SPX_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st) return st;
    const WsHeader *h = static_cast<const WsHeader *>(scratch);
    return record_launch(cudaMemcpyAsync(status, &h->status, sizeof(int32_t), cudaMemcpyDefault,
                                         reinterpret_cast<cudaStream_t>(stream)));
}
