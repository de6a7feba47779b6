// Shared device helpers and internal launcher declarations for the sm_103a
// dispatch / combine library.  The public C ABI is include/ep.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

// Record a data-dependent error: the status word keeps the largest code seen.
__device__ __forceinline__ void raise_status(int32_t *status, int code) {
    atomicMax(status, code);
}

// Every mbarrier wait in the library gives up after this many SM clocks
// (about a second) and reports EP_ERR_TIMEOUT instead of hanging.
constexpr long long kWaitLimit = 1LL << 31;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Make this thread's generic-proxy shared-memory writes visible to the TMA (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
// Make barrier initialisation visible to the other threads (of the cluster)
// and to the TMA.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
}
// Bounded wait for the phase of parity `parity` of a barrier (the phase
// before the current one counts as complete): false once `limit` SM clocks
// have passed, or as soon as *fail is set (when given).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *fail,
                                          long long limit = kWaitLimit) {
    const uint32_t a = smem_addr(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((fail && *fail) || clock64() - t0 > limit) return false;
    }
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Streaming 16-byte load of data read exactly once (no L1 allocation), through
// the non-coherent path: only for data that no kernel still running can write.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Streaming 16-byte load (no L1 allocation) on the coherent path, for data
// read once that must stay in flight across later stores: the assembler may
// move a non-coherent load below a store (it knows the data is read-only),
// which would serialise a "load the next row, store this one" loop; a coherent
// load may alias the store and keeps its place.
__device__ __forceinline__ uint4 ld_stream_coh(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Loads of what a programmatic predecessor wrote, issued after
// griddepcontrol.wait.  A const __restrict__ pointer or __ldg lets the
// compiler treat the data as read-only for the whole kernel (non-coherent
// loads, scheduled freely), which would let the load run before the wait and
// see the previous contents; a volatile asm load with a memory clobber stays
// after the wait and is a coherent (weak) global load.
__device__ __forceinline__ int32_t ld_dep(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float ld_dep(const float *p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_dep_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// Streaming (no L1 allocation) form of ld_dep_v4, for rows read exactly once.
__device__ __forceinline__ uint4 ld_dep_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Two packed bf16 -> two fp32 (exact: bf16 is the top half of binary32).
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Exclusive scan over n values produced by value(i), by one CTA of NT threads:
// out[i] = value(0) + ... + value(i-1) for i in [0, n], out[n] = total.  Thread t
// owns the contiguous run [t*ipt, (t+1)*ipt), ipt = ceil(n/NT).  `tmp` holds
// NT/32 ints of shared memory.  Must be reached by every thread of the CTA.
template <int NT, typename F>
__device__ __forceinline__ void block_exclusive_scan(int n, F value, int32_t *out,
                                                     int32_t *tmp) {
    static_assert(NT % 32 == 0 && NT / 32 <= 32, "one warp scans the warp totals");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ipt = (n + NT - 1) / NT;
    const int b0 = min(n, (int)threadIdx.x * ipt);
    const int b1 = min(n, b0 + ipt);
    int s = 0;
    for (int i = b0; i < b1; ++i) s += value(i);
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < NT / 32 ? tmp[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int o = __shfl_up_sync(kFullMask, wi, d);
            if (lane >= d) wi += o;
        }
        if (lane < NT / 32) tmp[lane] = wi - wv;
    }
    __syncthreads();
    const int excl = tmp[warp] + incl - s;
    int run = excl;
    for (int i = b0; i < b1; ++i) {
        out[i] = run;
        run += value(i);
    }
    if (threadIdx.x == NT - 1) out[n] = excl + s;  // runs past n are empty: this is the total
    __syncthreads();
}

// Per-device properties, cached on first use (host side).
int sm_count();

// An NVTX range named after the entry point around every C-ABI call, when
// the environment variable EP_NVTX=1 (read once per process); off by
// default.  Without a tool attached (nsys, ncu) NVTX calls do nothing.
bool trace_enabled();
struct TraceRange {
    explicit TraceRange(const char *name);
    ~TraceRange();
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
    bool on;
};

// Let kernel `k` take `dynamic` bytes of dynamic shared memory.  Without an
// explicit limit a CTA gets 48 KB of shared memory in all, the kernel's static
// shared memory included, so the limit is raised whenever the two together
// exceed that.
template <typename Kern>
cudaError_t allow_dynamic_smem(Kern k, size_t dynamic) {
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, k);
    if (err != cudaSuccess) return err;
    if (dynamic + fa.sharedSizeBytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dynamic);
}

// Launch with cudaLaunchKernelEx; `programmatic` lets the kernel start while the
// previous kernel on the stream still runs (programmatic dependent launch): it
// must then call griddepcontrol.wait before touching that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), int grid, int threads, size_t smem,
                          cudaStream_t stream, bool programmatic, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Internal launchers (one translation unit each).  They assume arguments were
// validated by the C ABI layer in abi.cu.
struct LayoutPlan {
    int threads;      // threads of the assign kernel's CTAs
    int chunk;        // entries per warp per pass
    int passes;       // passes per tile
    int tiles;        // tiles of topk_idx entries (CTAs that assign slots)
    int tile;         // entries per tile
    int grid;         // CTAs of the assign kernel (>= tiles; extra CTAs fill padding)
    size_t smem;      // dynamic shared memory of the assign kernel
    size_t ws_bytes;  // scratch: tiles x E int32 per-tile histograms (0 for the cluster kernel)
    bool cluster;     // decode-sized: one kernel of thread-block clusters (tiles = the CTAs of
                      // one, for the largest cluster; the launch may use fewer, larger slices)
};
LayoutPlan layout_plan(const ep_layout_t &L);
// Every argument check of ep_layout except the workspace's, in its order.
ep_status_t check_layout_call(const int32_t *topk_idx, const ep_layout_t *L);
cudaError_t launch_layout(const int32_t *topk_idx, const ep_layout_t &L, int32_t *workspace,
                          cudaStream_t stream);

// One CTA waiting on a barrier nothing completes, for at most limit_clocks.
cudaError_t launch_wait_selftest(int32_t *status, long long limit_clocks, cudaStream_t stream);
cudaError_t launch_cluster_wait_selftest(int32_t *status, long long limit_clocks,
                                         cudaStream_t stream);
// ep_layout followed by ep_dispatch, launched back to back.
cudaError_t launch_layout_dispatch(const int32_t *topk_idx, const ep_layout_t &L,
                                   int32_t *workspace, const void *x, int H, ep_quant_t quant,
                                   void *out_rows, void *out_scales, const float *topk_w,
                                   float *row_w, cudaStream_t stream);
cudaError_t launch_dispatch(const ep_layout_t &L, const void *x, int H, ep_quant_t quant,
                            void *out_rows, void *out_scales, const float *topk_w,
                            float *row_w, cudaStream_t stream);

cudaError_t launch_combine(const ep_layout_t &L, const void *y, int H, const float *topk_w,
                           void *out, cudaStream_t stream);

cudaError_t launch_masked_repack(const ep_layout_t &L, const void *rows,
                                 const void *row_scales, int H, ep_quant_t quant, int cap,
                                 void *slab, void *slab_scales, int32_t *masked_m,
                                 cudaStream_t stream);

cudaError_t launch_route(const float *logits, const float *bias, int T, int E, int K, int mode,
                         int n_group, int topk_group, int32_t *topk_idx, float *topk_w,
                         cudaStream_t stream);
cudaError_t launch_rank_ids(const int32_t *topk_idx, int T, int K, int E, int R,
                            int32_t *rank_idx, cudaStream_t stream);
cudaError_t launch_rank_expand(const ep_layout_t &rank_layout, const ep_layout_t &layout,
                               const int32_t *topk_idx, int row_bytes, int scale_bytes,
                               const void *send_rows, const void *send_scales, void *out_rows,
                               void *out_scales, cudaStream_t stream);

}  // namespace ep
