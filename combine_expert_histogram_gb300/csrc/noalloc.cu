// ep_layout_noalloc: ep_layout for callers that cannot allocate device memory.
//
// ep_layout needs scratch (per-tile expert histograms) that the caller
// normally passes in.  Some callers cannot provide it: a serving runtime that
// reserves all device memory at start-up and forbids allocation afterwards, a
// plugin that a host framework hands only its input and output buffers, or C
// code with no device allocator at hand.  This entry point takes its scratch
// from a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable of EP_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it names
// a stand-in object), so the first call on each device looks the address up
// with cudaGetSymbolAddress while that device is current, checks the result
// and caches it; that first call should therefore come before any stream
// capture.  All calls share the one array, which keeps whatever the last call
// left in it; every scratch word the layout kernels read is first written by
// the same call, so nothing has to be cleared.  Two calls whose work overlaps
// on the GPU (different streams, no ordering between them) race on the array.
#include <mutex>

#include "ep_common.cuh"

namespace {

__device__ __align__(256) int32_t g_layout_scratch[EP_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_layout_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ep_status_t ep_layout_noalloc(const int32_t *topk_idx, const ep_layout_t *layout,
                                         ep_stream_t stream) {
    const size_t need = ep_layout_workspace_bytes(layout);
    if (layout == nullptr) return EP_ERR_INVALID_ARG;
    if (need > EP_NOALLOC_SCRATCH_BYTES) return EP_ERR_CAPACITY;  // beyond the fixed array
    void *scratch = nullptr;
    if (need > 0 && scratch_address(&scratch) != cudaSuccess) return EP_ERR_CUDA;
    return ep_layout(topk_idx, layout, scratch, need, stream);
}
