// moe_dispatch_layout_noalloc: the dispatch layout for callers that cannot
// hand the library a workspace.
//
// Some callers have no way to allocate device memory when they call us: an
// inference runtime's plugin/enqueue path that forbids allocation while the
// network executes, or a host application whose device memory is owned entirely
// by its own pool and that cannot carve out a scratch buffer for a library.
// For them this entry point takes its scratch (per-block counts, slot starts,
// error word) from a file-scope __device__ array instead of a caller-provided
// workspace, and calls no cudaMalloc, cudaFree or allocating library routine.
//
// Limits and caveats:
//  - The array is kStaticScratchBytes (1 MiB) per GPU, held by every GPU that
//    loads the library until the process exits.  Shapes whose workspace
//    (moe_workspace_bytes) exceeds it are rejected with MOE_ERR_WORKSPACE.
//  - All calls on one GPU share the array, which keeps the last call's
//    contents.  Calls that overlap on the GPU (concurrent streams, several host
//    threads) race on it; serialise them.
//  - The first call on a device resolves the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current); make
//    that first call before any stream capture.  The address is kept for the
//    life of the process: after cudaDeviceReset on a device it no longer names
//    the array, so do not call this entry point on that device again.
//  - The error word at the start of the array is cleared at the start of every
//    call.  Device-detected input problems (ids out of range, a placement that
//    is not a permutation) are recorded there but not reported to the caller,
//    who has no handle on it: pass ids from moe_route and a valid permutation.
//    Every access stays in bounds either way.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device (set-up on first use).
moe_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_layout_noalloc(const int32_t* topk_ids,
                                                  const int32_t* placement,
                                                  const moe_shape* shape,
                                                  const moe_layout* layout, void* stream) {
    if (!shape) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_workspace_bytes(shape);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > moe::kStaticScratchBytes) return MOE_ERR_WORKSPACE;
    void* scratch = nullptr;
    const moe_status st = moe::scratch_address(&scratch);
    if (st != MOE_OK) return st;
    // only the error word must start at zero; the kernels write every count they read
    if (cudaMemsetAsync(scratch, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_dispatch_layout(topk_ids, placement, shape, layout, scratch,
                               moe::kStaticScratchBytes, stream);
}
