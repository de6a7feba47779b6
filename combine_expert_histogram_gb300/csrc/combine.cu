// ep_combine kernel: top-k weighted reduction of expert outputs back to token
// order ("weighted reduction in combine", vLLM tools/ep_kernels deepep_v2
// commit; combine reuses the dispatch handle, SGLang PR "moe: add DeepEP V2
// ElasticBuffer support to MoE token dispatcher", section "Motivation").
//
// out[t, h] = bf16_rn( sum_{k ascending, dst_row[t,k] >= 0} w[t,k] * y[dst_row[t,k], h] )
// with fp32 products and sums each rounded separately (__fmul_rn / __fadd_rn,
// so no fused multiply-add), starting from +0.
//
// HBM-bound gather: one lane owns 8 output elements (16 bytes) of one token;
// a warp covers 256 consecutive elements, so each of its K row loads is 512
// contiguous bytes.  The lane first issues all loads of a batch of 8 entries
// (8 x 16 B in flight per lane), then reduces them in k order.
#include <cuda_bf16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint16_t *y, int K, int H, long long n_chunks, const int32_t *dst_row,
                   const float *topk_w, uint16_t *__restrict__ out) {
    // Launched as a programmatic dependent: wait for the previous kernel on
    // the stream (it may have produced y) before reading anything.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long c = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (c >= n_chunks) return;
    const int CH = H >> 3;
    const int t = (int)(c / CH);
    const int j = (int)(c - (long long)t * CH);
    const int32_t *drow = dst_row + (size_t)t * K;
    const float *wrow = topk_w + (size_t)t * K;

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += kBatch) {
        int d[kBatch];
        float w[kBatch];
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int k = k0 + u;
            d[u] = k < K ? ld_dep(drow + k) : -1;
            w[u] = k < K ? ld_dep(wrow + k) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            v[u] = d[u] >= 0 ? ld_dep_stream(y + (size_t)d[u] * H + j * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (d[u] < 0) continue;
            const uint32_t p[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w[u], bf16_lo(p[i])));
                acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w[u], bf16_hi(p[i])));
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t *>(&b);  // .x (first) in the low half
    }
    st_v4(out + (size_t)t * H + j * 8, make_uint4(o[0], o[1], o[2], o[3]));
}

}  // namespace

cudaError_t launch_combine(const ep_layout_t &L, const void *y, int H, const float *topk_w,
                           void *out, cudaStream_t stream) {
    const int T = L.num_tokens, K = L.num_topk;
    if (T == 0) return cudaSuccess;
    const long long n = (long long)T * (H / 8);
    const long long blocks = (n + kThreads - 1) / kThreads;
    return launch_kernel(combine_kernel, (int)blocks, kThreads, 0, stream, true,
                         static_cast<const uint16_t *>(y), K, H, n, L.dst_row, topk_w,
                         static_cast<uint16_t *>(out));
}

}  // namespace ep
