// ep_dispatch kernels: scatter token rows into the layout, fused with dynamic
// 1x128 FP8-E4M3 quantisation (fp32 or packed UE8M0 scales).
//
// Format and scale conventions follow SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend" ("Supported scope": dynamic blockwise FP8;
// "Implementation": Hopper FP32 scales and Blackwell packed UE8M0 scales) and
// the vLLM tools/ep_kernels deepep_v2 commit ("FP8 block-quantized dispatch").
//
// HBM-bound: each token row is read once and written K times.  Work mapping:
//   FP8:  8 lanes own one 128-element group (16 bf16 = 32 B per lane, two
//         16-byte loads); a warp covers 4 consecutive groups; the group amax
//         is reduced with three xor-shuffles inside the 8 lanes; each lane
//         converts its 16 values to 16 E4M3 bytes and stores them as one
//         16-byte vector to each of the K destination rows, so every warp
//         store is 512 contiguous bytes.
//   bf16: one lane per 16-byte chunk; K 16-byte stores.
#include <cuda_fp8.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
    // __nv_cvt_float2_to_fp8x2: round to nearest even, saturate to +-448;
    // the first element of the pair lands in the low byte.
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

template <int Q>
__global__ void __launch_bounds__(kThreads)
    dispatch_fp8_kernel(const uint16_t *__restrict__ x, int K, int H, long long n_groups,
                        const int32_t *__restrict__ dst_row, uint8_t *__restrict__ out,
                        void *__restrict__ scales, const float *__restrict__ topk_w,
                        float *__restrict__ row_w) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 7;
    const long long grp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 3;
    if (grp >= n_groups) return;  // whole 8-lane groups leave together
    const unsigned gmask = 0xffu << (lane & 24);
    const int G = H >> 7;
    const int t = (int)(grp / G);
    const int g = (int)(grp - (long long)t * G);

    const uint16_t *src = x + (size_t)t * H + g * 128 + sub * 16;
    const uint4 a = ld_stream(src);
    const uint4 b = ld_stream(src + 8);
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
    uint32_t ebyte = 0;
    if (Q == EP_QUANT_FP8_F32) {
        q.x = fp8x4(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s), __fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
        q.y = fp8x4(__fdiv_rn(v[4], s), __fdiv_rn(v[5], s), __fdiv_rn(v[6], s), __fdiv_rn(v[7], s));
        q.z = fp8x4(__fdiv_rn(v[8], s), __fdiv_rn(v[9], s), __fdiv_rn(v[10], s), __fdiv_rn(v[11], s));
        q.w = fp8x4(__fdiv_rn(v[12], s), __fdiv_rn(v[13], s), __fdiv_rn(v[14], s), __fdiv_rn(v[15], s));
    } else {
        // scale rounded up to a power of two 2^(e-127); multiply by 2^(127-e)
        const uint32_t bits = __float_as_uint(s);
        const int e = (int)((bits >> 23) & 0xffu) + ((bits & 0x7fffffu) != 0u);
        const float inv = __uint_as_float((uint32_t)(254 - e) << 23);
        q.x = fp8x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
        q.y = fp8x4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
        q.z = fp8x4(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv), __fmul_rn(v[10], inv), __fmul_rn(v[11], inv));
        q.w = fp8x4(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv), __fmul_rn(v[14], inv), __fmul_rn(v[15], inv));
        ebyte = (uint32_t)e;
    }

    // UE8M0 with H a multiple of 512: the warp's 4 groups are bytes 0..3 of
    // one int32 scale word of one token; lane 0 packs and stores it.
    const bool packed_word = Q == EP_QUANT_FP8_UE8M0 && (G & 3) == 0;
    uint32_t word = 0;
    if (packed_word) {
        const uint32_t e1 = __shfl_sync(kFullMask, ebyte, 8);
        const uint32_t e2 = __shfl_sync(kFullMask, ebyte, 16);
        const uint32_t e3 = __shfl_sync(kFullMask, ebyte, 24);
        word = ebyte | (e1 << 8) | (e2 << 16) | (e3 << 24);
    }
    const int P4 = ((G + 3) >> 2) * 4;  // scale bytes per row, UE8M0

    const int32_t *drow = dst_row + (size_t)t * K;
    for (int k = 0; k < K; ++k) {
        const int d = __ldg(drow + k);
        if (d < 0) continue;
        st_v4(out + (size_t)d * H + g * 128 + sub * 16, q);
        if (sub == 0) {
            if (Q == EP_QUANT_FP8_F32) {
                reinterpret_cast<float *>(scales)[(size_t)d * G + g] = s;
            } else if (packed_word) {
                if (lane == 0) reinterpret_cast<uint32_t *>(scales)[(size_t)d * (P4 >> 2) + (g >> 2)] = word;
            } else {
                uint8_t *srow = reinterpret_cast<uint8_t *>(scales) + (size_t)d * P4;
                srow[g] = (uint8_t)ebyte;
                if (g == G - 1)
                    for (int p = G; p < P4; ++p) srow[p] = 127;  // 2^0 in unused bytes
            }
            if (row_w && g == 0) row_w[d] = __ldg(topk_w + (size_t)t * K + k);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    dispatch_bf16_kernel(const uint16_t *__restrict__ x, int K, int H, long long n_chunks,
                         const int32_t *__restrict__ dst_row, uint16_t *__restrict__ out,
                         const float *__restrict__ topk_w, float *__restrict__ row_w) {
    const long long c = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (c >= n_chunks) return;
    const int CH = H >> 3;
    const int t = (int)(c / CH);
    const int j = (int)(c - (long long)t * CH);
    const uint4 v = ld_stream(x + (size_t)t * H + j * 8);
    const int32_t *drow = dst_row + (size_t)t * K;
    for (int k = 0; k < K; ++k) {
        const int d = __ldg(drow + k);
        if (d < 0) continue;
        st_v4(out + (size_t)d * H + j * 8, v);
        if (row_w && j == 0) row_w[d] = __ldg(topk_w + (size_t)t * K + k);
    }
}

}  // namespace

cudaError_t launch_dispatch(const ep_layout_t &L, const void *x, int H, ep_quant_t quant,
                            void *out_rows, void *out_scales, const float *topk_w,
                            float *row_w, cudaStream_t stream) {
    const int T = L.num_tokens, K = L.num_topk;
    if (T == 0) return cudaSuccess;
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    if (quant == EP_QUANT_NONE) {
        const long long n = (long long)T * (H / 8);
        const long long blocks = (n + kThreads - 1) / kThreads;
        dispatch_bf16_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
            xb, K, H, n, L.dst_row, static_cast<uint16_t *>(out_rows), topk_w, row_w);
    } else {
        const long long n = (long long)T * (H / 128);
        const long long blocks = (n * 8 + kThreads - 1) / kThreads;
        uint8_t *o = static_cast<uint8_t *>(out_rows);
        if (quant == EP_QUANT_FP8_F32)
            dispatch_fp8_kernel<EP_QUANT_FP8_F32><<<(unsigned)blocks, kThreads, 0, stream>>>(
                xb, K, H, n, L.dst_row, o, out_scales, topk_w, row_w);
        else
            dispatch_fp8_kernel<EP_QUANT_FP8_UE8M0><<<(unsigned)blocks, kThreads, 0, stream>>>(
                xb, K, H, n, L.dst_row, o, out_scales, topk_w, row_w);
    }
    return cudaGetLastError();
}

}  // namespace ep
