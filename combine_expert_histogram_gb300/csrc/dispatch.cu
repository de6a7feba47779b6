// ep_dispatch kernels: scatter token rows into the layout, fused with dynamic
// 1x128 FP8-E4M3 quantisation (fp32 or packed UE8M0 scales) or 1x32 MXFP8.
//
// Format and scale conventions follow SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend" ("Supported scope": dynamic blockwise FP8;
// "Implementation": Hopper FP32 scales and Blackwell packed UE8M0 scales) and
// the vLLM tools/ep_kernels deepep_v2 commit ("FP8 block-quantized dispatch");
// MXFP8 is the "1x32 MXFP8 ... with dynamic activation scaling" format of the
// SGLang discussion "deepep v2 support?", scaled by the OCP Microscaling (MX)
// v1.0 rule X = 2^(floor(log2 amax) - 8).
//
// HBM-bound: each token row is read once and written K times (80 % of the
// bytes are writes).  One CTA owns one token:
//   1. its threads load the row (16 bf16 = two 16-byte loads per thread),
//      8 consecutive lanes per 128-element group; the group amax is reduced
//      with three xor-shuffles inside those 8 lanes;
//   2. each thread converts its 16 values to E4M3 and writes them, with the
//      group's scale, into a shared-memory copy of the output row;
//   3. after a proxy fence, a wait for the layout kernels (dispatch is
//      launched as their programmatic dependent, so steps 1-2 overlap them)
//      and a barrier, one thread issues one
//      cp.async.bulk store per destination row (the whole H-byte row, and the
//      fp32 scale row when its size is a multiple of 16 bytes), so the TMA
//      engine writes K contiguous rows while the SM moves on;
//   4. the thread waits for the bulk stores to finish reading shared memory
//      before the CTA exits.
// Scale rows that are not a multiple of 16 bytes (packed UE8M0, or fp32 with
// H/128 not a multiple of 4) are written by plain 4-byte stores.
#include <cuda_fp8.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kMaxThreads = 512;

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
    // __nv_cvt_float2_to_fp8x2: round to nearest even, saturate to +-448;
    // the first element of the pair lands in the low byte.
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// shared memory to global memory, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the TMA (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int Q>
__global__ void __launch_bounds__(kMaxThreads)
    dispatch_kernel(const uint16_t *__restrict__ x, int K, int H,
                    const int32_t *__restrict__ dst_row, uint8_t *__restrict__ out,
                    void *__restrict__ scales, const float *__restrict__ topk_w,
                    float *__restrict__ row_w, bool bulk_scales, int mn_stride, int mn_cap) {
    // bulk_scales: fp32 scale rows are a multiple of 16 bytes and `scales` is
    // 16-byte aligned, so they go out with the TMA too
    extern __shared__ __align__(128) uint8_t stage[];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int G = H >> 7;
    // staged bytes: the row (H fp8 or 2H bf16), then the scale row
    const int row_bytes = Q == EP_QUANT_NONE ? 2 * H : H;
    const int P4 = ((G + 3) >> 2) * 4;  // UE8M0 scale bytes per row
    constexpr bool kUe8m0 = Q == EP_QUANT_FP8_UE8M0 || Q == EP_QUANT_FP8_UE8M0_MN;
    const int scale_bytes = (Q == EP_QUANT_FP8_F32 || Q == EP_QUANT_MXFP8) ? 4 * G
                            : kUe8m0 ? P4 : 0;
    uint8_t *srow = stage;
    uint8_t *sscale = stage + row_bytes;
    __shared__ int32_t sdst[EP_MAX_TOPK];

    if (kUe8m0 && threadIdx.x < P4 - G) sscale[G + threadIdx.x] = 127;  // 2^0

    const uint16_t *xr = x + (size_t)t * H;
    if (Q == EP_QUANT_NONE) {
        for (int j = threadIdx.x; j < H / 8; j += blockDim.x)
            reinterpret_cast<uint4 *>(srow)[j] = ld_stream(xr + j * 8);
    } else {
        // slot j: group j/8, elements (j%8)*16 .. +15 of that group
        for (int j = threadIdx.x; j < G * 8; j += blockDim.x) {  // block-uniform trip count per warp
            const int g = j >> 3, sub = j & 7;
            const unsigned gmask = 0xffu << (lane & 24);
            const uint4 a = ld_stream(xr + g * 128 + sub * 16);
            const uint4 b = ld_stream(xr + g * 128 + sub * 16 + 8);
            float v[16];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[2 * i] = bf16_lo(w[i]);
                v[2 * i + 1] = bf16_hi(w[i]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
            amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 4));
            amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
            // s = max(amax, 1e-4) / 448, an IEEE round-to-nearest division.
            const float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
            uint4 q;
            if (Q == EP_QUANT_FP8_F32) {
                q.x = fp8x4(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s), __fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
                q.y = fp8x4(__fdiv_rn(v[4], s), __fdiv_rn(v[5], s), __fdiv_rn(v[6], s), __fdiv_rn(v[7], s));
                q.z = fp8x4(__fdiv_rn(v[8], s), __fdiv_rn(v[9], s), __fdiv_rn(v[10], s), __fdiv_rn(v[11], s));
                q.w = fp8x4(__fdiv_rn(v[12], s), __fdiv_rn(v[13], s), __fdiv_rn(v[14], s), __fdiv_rn(v[15], s));
                if (sub == 0) reinterpret_cast<float *>(sscale)[g] = s;
            } else if (Q == EP_QUANT_MXFP8) {
                // two lanes hold one 32-element block: X = 2^(floor(log2 amax) - 8),
                // clamped at 2^-127; byte = log2(X) + 127; multiply by 1/X = 2^(127-byte)
                float bmax = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
                bmax = fmaxf(bmax, __shfl_xor_sync(gmask, bmax, 1));
                const int be = (int)((__float_as_uint(bmax) >> 23) & 0xffu);  // 0: zero/subnormal
                const int byte = be > 8 ? be - 8 : 0;
                const float inv = __uint_as_float((uint32_t)(254 - byte) << 23);
                q.x = fp8x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
                q.y = fp8x4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
                q.z = fp8x4(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv), __fmul_rn(v[10], inv), __fmul_rn(v[11], inv));
                q.w = fp8x4(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv), __fmul_rn(v[14], inv), __fmul_rn(v[15], inv));
                if ((sub & 1) == 0) sscale[g * 4 + (sub >> 1)] = (uint8_t)byte;
            } else {
                // scale rounded up to a power of two 2^(e-127); multiply by 2^(127-e)
                const uint32_t bits = __float_as_uint(s);
                const int e = (int)((bits >> 23) & 0xffu) + ((bits & 0x7fffffu) != 0u);
                const float inv = __uint_as_float((uint32_t)(254 - e) << 23);
                q.x = fp8x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
                q.y = fp8x4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
                q.z = fp8x4(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv), __fmul_rn(v[10], inv), __fmul_rn(v[11], inv));
                q.w = fp8x4(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv), __fmul_rn(v[14], inv), __fmul_rn(v[15], inv));
                if (sub == 0) sscale[g] = (uint8_t)e;
            }
            reinterpret_cast<uint4 *>(srow)[j] = q;
        }
    }
    fence_proxy_async_smem();
    // x was complete before the layout started; dst_row is the layout's
    // output: wait for it (a no-op without a programmatic edge).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < K) sdst[threadIdx.x] = dst_row[(size_t)t * K + threadIdx.x];
    __syncthreads();

    // one thread hands the staged row to the TMA engine, once per destination
    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            const int d = sdst[k];
            if (d < 0) continue;
            bulk_store(out + (size_t)d * row_bytes, srow, (uint32_t)row_bytes);
            if (bulk_scales)
                bulk_store(static_cast<uint8_t *>(scales) + (size_t)d * scale_bytes, sscale,
                           (uint32_t)scale_bytes);
        }
        bulk_commit();
    }
    // remaining scale rows: 4-byte words by the other threads (row-major, or
    // MN-major: word wd of row d at wd*stride + d, per expert for masked)
    if (Q != EP_QUANT_NONE && !bulk_scales) {
        const int words = Q == EP_QUANT_NONE ? 1 : scale_bytes >> 2;  // (bf16 never gets here)
        for (int j = threadIdx.x; j < K * words; j += blockDim.x) {
            const int k = j / words, wd = j - k * words;
            const int d = sdst[k];
            if (d < 0) continue;
            size_t at = (size_t)d * words + wd;
            if (Q == EP_QUANT_FP8_UE8M0_MN)
                at = mn_cap ? ((size_t)(d / mn_cap) * words + wd) * mn_stride + (size_t)(d % mn_cap)
                            : (size_t)wd * mn_stride + d;
            reinterpret_cast<uint32_t *>(scales)[at] = reinterpret_cast<const uint32_t *>(sscale)[wd];
        }
    }
    if (row_w && threadIdx.x < K) {
        const int d = sdst[threadIdx.x];
        if (d >= 0) row_w[d] = __ldg(topk_w + (size_t)t * K + threadIdx.x);
    }
    if (threadIdx.x == 0) bulk_wait_read();  // staging must outlive the bulk reads
}

template <int Q>
cudaError_t launch_q(const ep_layout_t &L, const void *x, int H, void *out_rows,
                     void *out_scales, const float *topk_w, float *row_w, cudaStream_t stream) {
    const int G = H / 128;
    const int row_bytes = Q == EP_QUANT_NONE ? 2 * H : H;
    const int scale_bytes = (Q == EP_QUANT_FP8_F32 || Q == EP_QUANT_MXFP8) ? 4 * G
                            : (Q == EP_QUANT_FP8_UE8M0 || Q == EP_QUANT_FP8_UE8M0_MN) ? ((G + 3) / 4) * 4
                            : 0;
    const size_t smem = (size_t)row_bytes + (size_t)scale_bytes;
    // one slot per 16 elements (FP8) or per 16-byte chunk (bf16), up to 512 threads
    int slots = Q == EP_QUANT_NONE ? H / 8 : G * 8;
    int threads = ((slots + 31) / 32) * 32;
    if (threads > kMaxThreads) threads = kMaxThreads;
    if (threads < 64) threads = 64;  // K <= 32 threads read dst_row; scale pads
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(dispatch_kernel<Q>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    const bool bulk_scales = (Q == EP_QUANT_FP8_F32 || Q == EP_QUANT_MXFP8) &&
                             (scale_bytes % 16) == 0 &&
                             (reinterpret_cast<uintptr_t>(out_scales) % 16) == 0;
    // programmatic dependent of the layout: x is loaded and quantised while
    // the layout kernels finish
    // MN-major scale columns: padded row space (contiguous) or padded capacity per expert
    const bool masked = L.kind == EP_LAYOUT_MASKED;
    const long long rows_cap = masked ? (long long)L.num_experts * L.capacity
                                      : (long long)L.num_tokens * L.num_topk +
                                            (long long)(L.num_tokens * L.num_topk < L.num_experts
                                                            ? L.num_tokens * L.num_topk
                                                            : L.num_experts) * (L.align - 1);
    const int mn_cap = masked ? L.capacity : 0;
    const int mn_stride = masked ? (L.capacity + 3) / 4 * 4 : (int)((rows_cap + 3) / 4 * 4);
    return launch_kernel(dispatch_kernel<Q>, L.num_tokens, threads, smem, stream, true,
                         static_cast<const uint16_t *>(x), L.num_topk, H, L.dst_row,
                         static_cast<uint8_t *>(out_rows), out_scales, topk_w, row_w,
                         bulk_scales, mn_stride, mn_cap);
}

}  // namespace

cudaError_t launch_dispatch(const ep_layout_t &L, const void *x, int H, ep_quant_t quant,
                            void *out_rows, void *out_scales, const float *topk_w,
                            float *row_w, cudaStream_t stream) {
    if (L.num_tokens == 0) return cudaSuccess;
    switch (quant) {
        case EP_QUANT_NONE:
            return launch_q<EP_QUANT_NONE>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        case EP_QUANT_FP8_F32:
            return launch_q<EP_QUANT_FP8_F32>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        case EP_QUANT_MXFP8:
            return launch_q<EP_QUANT_MXFP8>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        case EP_QUANT_FP8_UE8M0_MN:
            return launch_q<EP_QUANT_FP8_UE8M0_MN>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        default:
            return launch_q<EP_QUANT_FP8_UE8M0>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
    }
}

}  // namespace ep
