// ep_combine kernel: top-k weighted reduction of expert outputs back to token
// order ("weighted reduction in combine", vLLM tools/ep_kernels deepep_v2
// commit; combine reuses the dispatch handle, SGLang PR "moe: add DeepEP V2
// ElasticBuffer support to MoE token dispatcher", section "Motivation").
//
// out[t, h] = bf16_rn( sum_{k ascending, dst_row[t,k] >= 0} w[t,k] * y[dst_row[t,k], h] )
// with fp32 products and sums each rounded separately (no fused multiply-add),
// starting from +0.  The products come two at a time from packed f32x2
// multiplies (each lane an IEEE round-to-nearest multiply); the sums stay
// scalar __fadd_rn: with a packed add consuming a packed product, the pair is
// contracted into a fused multiply-add (results then differ from separate
// rounding in cancelling sums).  Measured on GB300: the contraction happens
// in the assembler, for packed `add.rn.f32x2` after `mul.rn.f32x2` written
// as inline PTX with explicit rounding, after an `fma.rn.f32x2` with a -0
// addend, and with --fmad=false (each packed operation alone was exact; the
// chain differed from the scalar one in 43 % of 2 M random pairs).
//
// HBM-bound gather: one lane owns 8 output elements (16 bytes) of one token
// -- 16 elements with one 256-bit load per row when the batch fills the GPU
// (combine32_kernel) --; a warp covers 256 (512) consecutive elements, so
// each of its K row loads is 512 (1024) contiguous bytes.  The lane first issues all loads of a batch of 8 entries
// (8 x 16 B in flight per lane), then reduces them in k order.  The token's
// destinations and weights come as 16-byte loads where K allows.
#include <cuda_bf16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 128;
constexpr int kBatch = 8;

// Two fp32 lanes in one 64-bit register (element 0 in the low half), and the
// packed sm_100+ multiply on them: each lane is an IEEE round-to-nearest
// multiply, exactly what __fmul_rn gives per element.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float2 split_f32x2(uint64_t a) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a));
    return r;
}

// kVec: K is a multiple of 4 and dst_row / topk_w are 16-byte aligned, so a
// token's destinations and weights arrive as 16-byte loads (4 entries each)
// instead of one load per entry.
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint16_t *y, int K, int H, long long n_chunks, const int32_t *dst_row,
                   const float *topk_w, uint16_t *__restrict__ out) {
    // Launched as a programmatic dependent: wait for the previous kernel on
    // the stream (it may have produced y) before reading anything.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // whatever follows waits for this kernel itself: let it launch now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long c = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (c >= n_chunks) return;
    const int CH = H >> 3;
    const int t = (int)(c / CH);
    const int j = (int)(c - (long long)t * CH);
    const int32_t *drow = dst_row + (size_t)t * K;
    const float *wrow = topk_w + (size_t)t * K;

    uint64_t acc[4];  // output pairs (8i, 8i+1): fp32, from +0
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = 0;

    for (int k0 = 0; k0 < K; k0 += kBatch) {
        int d[kBatch];
        float w[kBatch];
        uint4 v[kBatch];
        if (kVec) {
#pragma unroll
            for (int q = 0; q < kBatch / 4; ++q) {
                const bool in = k0 + 4 * q < K;  // whole quads: K % 4 == 0
                const uint4 dq = in ? ld_dep_v4(drow + k0 + 4 * q) : make_uint4(~0u, ~0u, ~0u, ~0u);
                const uint4 wq = in ? ld_dep_v4(wrow + k0 + 4 * q) : make_uint4(0, 0, 0, 0);
                d[4 * q] = (int)dq.x, d[4 * q + 1] = (int)dq.y, d[4 * q + 2] = (int)dq.z,
                d[4 * q + 3] = (int)dq.w;
                w[4 * q] = __uint_as_float(wq.x), w[4 * q + 1] = __uint_as_float(wq.y),
                w[4 * q + 2] = __uint_as_float(wq.z), w[4 * q + 3] = __uint_as_float(wq.w);
            }
        } else {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + u;
                d[u] = k < K ? ld_dep(drow + k) : -1;
                w[u] = k < K ? ld_dep(wrow + k) : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            v[u] = d[u] >= 0 ? ld_dep_stream(y + (size_t)d[u] * H + j * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (d[u] < 0) continue;
            const uint64_t w2 = f32x2(w[u], w[u]);
            const uint32_t p[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 m = split_f32x2(mul_f32x2(w2, f32x2(bf16_lo(p[i]), bf16_hi(p[i]))));
                const float2 a = split_f32x2(acc[i]);
                acc[i] = f32x2(__fadd_rn(a.x, m.x), __fadd_rn(a.y, m.y));
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = split_f32x2(acc[i]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(a.x, a.y);
        o[i] = *reinterpret_cast<const uint32_t *>(&b);  // .x (first) in the low half
    }
    st_v4(out + (size_t)t * H + j * 8, make_uint4(o[0], o[1], o[2], o[3]));
}

// 32-byte lanes: one lane owns 16 outputs and reads 32 bytes of each row with
// one 256-bit load (evict-first in L2: every row is read once); batches of 4
// rows keep 128 bytes in flight per lane.  Needs H % 16 == 0 and 32-byte
// aligned y and out.
constexpr int kBatch32 = 4;

__device__ __forceinline__ void ld_row32(const void *p, uint32_t (&r)[8]) {
    asm volatile("ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "l"(p)
                 : "memory");
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    combine32_kernel(const uint16_t *y, int K, int H, long long n_chunks, const int32_t *dst_row,
                     const float *topk_w, uint16_t *__restrict__ out) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // whatever follows waits for this kernel itself: let it launch now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long c = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (c >= n_chunks) return;
    const int CH = H >> 4;  // 16-output chunks per token
    const int t = (int)(c / CH);
    const int j = (int)(c - (long long)t * CH);
    const int32_t *drow = dst_row + (size_t)t * K;
    const float *wrow = topk_w + (size_t)t * K;
    uint64_t acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    for (int k0 = 0; k0 < K; k0 += kBatch32) {
        int d[kBatch32];
        float w[kBatch32];
        if (kVec) {  // K % 4 == 0: one quad per batch
            const uint4 dq = ld_dep_v4(drow + k0);
            const uint4 wq = ld_dep_v4(wrow + k0);
            d[0] = (int)dq.x, d[1] = (int)dq.y, d[2] = (int)dq.z, d[3] = (int)dq.w;
            w[0] = __uint_as_float(wq.x), w[1] = __uint_as_float(wq.y);
            w[2] = __uint_as_float(wq.z), w[3] = __uint_as_float(wq.w);
        } else {
#pragma unroll
            for (int u = 0; u < kBatch32; ++u) {
                const int k = k0 + u;
                d[u] = k < K ? ld_dep(drow + k) : -1;
                w[u] = k < K ? ld_dep(wrow + k) : 0.0f;
            }
        }
        uint32_t v[kBatch32][8];
#pragma unroll
        for (int u = 0; u < kBatch32; ++u) {
            if (d[u] >= 0) {
                ld_row32(y + (size_t)d[u] * H + (size_t)j * 16, v[u]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[u][i] = 0;
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch32; ++u) {
            if (d[u] < 0) continue;
            const uint64_t w2 = f32x2(w[u], w[u]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 m = split_f32x2(mul_f32x2(w2, f32x2(bf16_lo(v[u][i]), bf16_hi(v[u][i]))));
                const float2 a = split_f32x2(acc[i]);
                acc[i] = f32x2(__fadd_rn(a.x, m.x), __fadd_rn(a.y, m.y));
            }
        }
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 a = split_f32x2(acc[i]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(a.x, a.y);
        o[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    uint16_t *op = out + (size_t)t * H + (size_t)j * 16;
    st_v4(op, make_uint4(o[0], o[1], o[2], o[3]));
    st_v4(op + 8, make_uint4(o[4], o[5], o[6], o[7]));
}

}  // namespace

cudaError_t launch_combine(const ep_layout_t &L, const void *y, int H, const float *topk_w,
                           void *out, cudaStream_t stream) {
    const int T = L.num_tokens, K = L.num_topk;
    if (T == 0) return cudaSuccess;
    const long long n = (long long)T * (H / 8);
    const long long blocks = (n + kThreads - 1) / kThreads;
    const bool vec = K % 4 == 0 && reinterpret_cast<uintptr_t>(L.dst_row) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(topk_w) % 16 == 0;
    // 32-byte lanes when there is enough work to fill the GPU with half the
    // threads (at least four CTAs per SM); small decode batches keep the
    // 16-byte lanes' wider grid
    const long long n32 = (long long)T * (H / 16);
    const long long b32 = (n32 + kThreads - 1) / kThreads;
    if (H % 16 == 0 && b32 >= 4LL * sm_count() && reinterpret_cast<uintptr_t>(y) % 32 == 0 &&
        reinterpret_cast<uintptr_t>(out) % 32 == 0) {
        return vec ? launch_kernel(combine32_kernel<true>, (int)b32, kThreads, 0, stream, true,
                                   static_cast<const uint16_t *>(y), K, H, n32, L.dst_row, topk_w,
                                   static_cast<uint16_t *>(out))
                   : launch_kernel(combine32_kernel<false>, (int)b32, kThreads, 0, stream, true,
                                   static_cast<const uint16_t *>(y), K, H, n32, L.dst_row, topk_w,
                                   static_cast<uint16_t *>(out));
    }
    return vec ? launch_kernel(combine_kernel<true>, (int)blocks, kThreads, 0, stream, true,
                               static_cast<const uint16_t *>(y), K, H, n, L.dst_row, topk_w,
                               static_cast<uint16_t *>(out))
               : launch_kernel(combine_kernel<false>, (int)blocks, kThreads, 0, stream, true,
                               static_cast<const uint16_t *>(y), K, H, n, L.dst_row, topk_w,
                               static_cast<uint16_t *>(out));
}

}  // namespace ep
