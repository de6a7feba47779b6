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
// capture.  The cached address belongs to the CUDA context it was looked up
// in: after cudaDeviceReset the runtime builds a new context, in which the
// array may sit elsewhere, so the cache also records the context's unique id
// and the address is looked up again when the current context differs.  All
// calls share the one array, which keeps whatever the last call left in it;
// every scratch word the layout kernels read is first written by the same
// call, so nothing has to be cleared.  Two calls whose work overlaps on the
// GPU (different streams, no ordering between them) race on the array.
#include <cuda.h>

#include <mutex>

#include "ep_common.cuh"

namespace {

__device__ __align__(256) int32_t g_layout_scratch[EP_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    unsigned long long ctx_id;  // unique id of the context the address belongs to
    void *ptr;                  // nullptr: not looked up yet
};

std::mutex g_mu;
ScratchSlot g_slot[kMaxDevices] = {};

// The driver's cuCtxGetCurrent and cuCtxGetId, reached through the runtime
// (the library links no driver library of its own).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

cudaError_t driver_fns(CtxGetCurrentFn *get_current, CtxGetIdFn *get_id) {
    static CtxGetCurrentFn cur = nullptr;
    static CtxGetIdFn id = nullptr;
    if (cur == nullptr || id == nullptr) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult r2 = cudaDriverEntryPointSymbolNotFound;
        cudaError_t err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000,
                                                           cudaEnableDefault, &r1);
        if (err != cudaSuccess) return err;
        err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2);
        if (err != cudaSuccess) return err;
        if (r1 != cudaDriverEntryPointSuccess || r2 != cudaDriverEntryPointSuccess || !p || !q)
            return cudaErrorSymbolNotFound;
        cur = reinterpret_cast<CtxGetCurrentFn>(p);
        id = reinterpret_cast<CtxGetIdFn>(q);
    }
    *get_current = cur;
    *get_id = id;
    return cudaSuccess;
}

// Unique id of the calling thread's current context (0 if none is current).
cudaError_t current_ctx_id(unsigned long long *out) {
    CtxGetCurrentFn get_current;
    CtxGetIdFn get_id;
    cudaError_t err = driver_fns(&get_current, &get_id);
    if (err != cudaSuccess) return err;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
    *out = 0;
    if (ctx != nullptr && get_id(ctx, out) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
    return cudaSuccess;
}

// Device address of g_layout_scratch in the current device's current context
// (looked up once per device and context).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    err = current_ctx_id(&id);
    if (err != cudaSuccess) return err;
    ScratchSlot &slot = g_slot[dev];
    if (slot.ptr == nullptr || id == 0 || slot.ctx_id != id) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_layout_scratch);  // makes the context current if needed
        if (err != cudaSuccess) return err;
        if (id == 0) {  // no context was current before the lookup: read the new one's id
            err = current_ctx_id(&id);
            if (err != cudaSuccess) return err;
        }
        slot.ptr = p;
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" ep_status_t ep_layout_noalloc(const int32_t *topk_idx, const ep_layout_t *layout,
                                         ep_stream_t stream) {
    const ep::TraceRange trace("ep_layout_noalloc");
    // ep_layout's own argument checks first, in its order, so that both calls
    // give the same code for the same bad arguments; the array's size next
    const ep_status_t st = ep::check_layout_call(topk_idx, layout);
    if (st != EP_OK) return st;
    const size_t need = ep_layout_workspace_bytes(layout);
    if (need > EP_NOALLOC_SCRATCH_BYTES) return EP_ERR_CAPACITY;  // beyond the fixed array
    void *scratch = nullptr;
    if (need > 0 && scratch_address(&scratch) != cudaSuccess) return EP_ERR_CUDA;
    return ep_layout(topk_idx, layout, scratch, need, stream);
}
