// fwd_noalloc.cu -- gdn_chunk_fwd_noalloc: the GDN chunk forward without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// forward: code that runs inside a CUDA-graph capture whose allocator is not
// graph-aware, runtimes that freeze their memory budget after start-up and
// forbid further cudaMalloc calls, and plugin hosts that hand out tensors but
// no allocator.  For them this entry point keeps the forward's scratch (the
// per-chunk [T diag(beta Gamma); T; L] matrices of the tensor-core path) in a
// fixed file-scope device array instead of the `workspace` field of
// gcl_fwd_args.  The launch plan is the fastest one whose scratch fits in the array
// (problems with few units whose transition-form records do not fit run the W form).  The array is part of the library image: every GPU that loads
// the library holds kNoallocScratchBytes of device memory until the process
// exits.  Problems whose scratch would not fit are rejected on the host.
//
// Set-up: the device address of the array is looked up with
// cudaGetSymbolAddress the first time the entry point runs on a device (with
// that device current) and cached per device; that first call should therefore
// be made before any stream capture begins.
//
// Every call on a device shares the one array and leaves its contents behind.
// Nothing in it has to start at zero: each call writes the scratch of every
// live chunk before reading it.  Calls whose executions overlap on the GPU
// (different streams without ordering, or concurrent graph replays) race on
// the array and must be avoided by the caller.
#include <mutex>

#include "gcl_internal.cuh"

namespace gcl {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on first use).
gcl_status_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_check(e, "gdn_chunk_fwd_noalloc (cudaGetDevice)");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GCL_ERR_UNSUPPORTED, "gdn_chunk_fwd_noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_check(e, "gdn_chunk_fwd_noalloc (cudaGetSymbolAddress)");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GCL_OK;
}

}  // namespace
}  // namespace gcl

using namespace gcl;

extern "C" size_t gcl_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }

extern "C" gcl_status_t gdn_chunk_fwd_noalloc(const gcl_fwd_args *args, gcl_stream_t stream) {
    if (!args) return fail(GCL_ERR_INVALID_ARG, "gdn_chunk_fwd_noalloc: args is NULL");
    const size_t need = gcl_fwd_workspace_min_bytes(args);
    if (need > kNoallocScratchBytes)
        return fail(GCL_ERR_CAPACITY,
                    "gdn_chunk_fwd_noalloc: these sizes need %zu bytes of scratch; the "
                    "library's static scratch holds %zu bytes (use gdn_chunk_fwd with a "
                    "caller workspace)",
                    need, kNoallocScratchBytes);
    gcl_fwd_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (need > 0) {
        gcl_status_t st = noalloc_scratch(&a.workspace);
        if (st != GCL_OK) return st;
        a.workspace_bytes = kNoallocScratchBytes;
    }
    return gdn_chunk_fwd(&a, stream);
}
