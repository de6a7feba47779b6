// ep_route_topk: router output (topk_idx, topk_w) from logits, the step before
// ep_layout (the topk_idx that V2 dispatch infers its layout from: SGLang PR
// "moe: add DeepEP V2 ElasticBuffer support to MoE token dispatcher",
// "Motivation"), for the two router families of the model list in SGLang PR
// "[Feature] Add DeepEPv2 (ElasticBuffer) MoE A2A backend", "Supported scope":
//   softmax:         top-K of softmax(logits) (= top-K of the logits, softmax
//                    being monotone), weights renormalised over the K picks;
//   grouped sigmoid: s = sigmoid(logit), c = s + bias; group score = sum of the
//                    two largest c of each group; keep the topk_group best
//                    groups; top-K of c inside them; weights s / sum(s).
// Ties go to the lower expert (or group) id.  Selection decisions are taken in
// fp32.
//
// One warp per token: the warp stages the token's scores in shared memory,
// lane g computes group g's score, and each of the K picks is a warp-wide
// argmax (lane-local scan, then five xor-shuffle rounds on (value, index)).
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kWarpsPerCta = 4;

__device__ __forceinline__ bool ranks_before(float va, int a, float vb, int b) {
    return va > vb || (va == vb && a < b);
}

// Warp-wide best (value, index) of sc[0..n) among lanes; every lane gets it.
__device__ __forceinline__ void warp_best(const float *sc, int n, float &bv, int &bi) {
    const int lane = threadIdx.x & 31;
    bv = -INFINITY;
    bi = 0x7fffffff;
    for (int e = lane; e < n; e += 32) {
        const float v = sc[e];
        if (ranks_before(v, e, bv, bi)) {
            bv = v;
            bi = e;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFullMask, bv, off);
        const int oi = __shfl_xor_sync(kFullMask, bi, off);
        if (ranks_before(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    route_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E,
                 int K, int n_group, int topk_group, int32_t *__restrict__ topk_idx,
                 float *__restrict__ topk_w) {
    extern __shared__ float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kWarpsPerCta + warp;
    if (t >= T) return;  // whole warps
    float *sc = smem + (size_t)warp * 2 * E;  // selection scores
    float *sg = sc + E;                       // logits (softmax) or sigmoids
    const float *l = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
        const float v = __ldg(l + e);
        if (MODE == EP_ROUTE_SOFTMAX) {
            sc[e] = v;
            sg[e] = v;
        } else {
            const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-v)));
            sg[e] = s;
            sc[e] = __fadd_rn(s, bias ? __ldg(bias + e) : 0.0f);
        }
    }
    __syncwarp();
    if (MODE == EP_ROUTE_GROUPED_SIGMOID) {
        const int gs = E / n_group;
        float gscore = -INFINITY;
        if (lane < n_group) {  // the two largest c of group `lane`, ties to the lower id
            float v1 = -INFINITY, v2 = -INFINITY;
            int i1 = 0x7fffffff, i2 = 0x7fffffff;
            for (int e = lane * gs; e < (lane + 1) * gs; ++e) {
                const float v = sc[e];
                if (ranks_before(v, e, v1, i1)) {
                    v2 = v1;
                    i2 = i1;
                    v1 = v;
                    i1 = e;
                } else if (ranks_before(v, e, v2, i2)) {
                    v2 = v;
                    i2 = e;
                }
            }
            gscore = __fadd_rn(v1, v2);
        }
        unsigned keep = 0;  // bit g: group g kept
        for (int j = 0; j < topk_group; ++j) {
            float bv = lane < n_group && !((keep >> lane) & 1u) ? gscore : -INFINITY;
            int bi = lane < n_group && !((keep >> lane) & 1u) ? lane : 0x7fffffff;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(kFullMask, bv, off);
                const int oi = __shfl_xor_sync(kFullMask, bi, off);
                if (ranks_before(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            keep |= 1u << bi;
        }
        for (int e = lane; e < E; e += 32)
            if (!((keep >> (e / gs)) & 1u)) sc[e] = -INFINITY;
        __syncwarp();
    }
    int my_pick = 0;
    for (int j = 0; j < K; ++j) {
        float bv;
        int bi;
        warp_best(sc, E, bv, bi);
        if (lane == j) my_pick = bi;
        __syncwarp();
        if (lane == 0) sc[bi] = -INFINITY;  // taken
        __syncwarp();
    }
    // weights over the K picks, lane j holds pick j
    float wv = 0.0f;
    if (MODE == EP_ROUTE_SOFTMAX) {
        const float top = __shfl_sync(kFullMask, lane < K ? sg[my_pick] : -INFINITY, 0);
        if (lane < K) wv = expf(__fadd_rn(sg[my_pick], -top));
    } else if (lane < K) {
        wv = sg[my_pick];
    }
    float sum = 0.0f;  // ascending j
    for (int j = 0; j < K; ++j) sum = __fadd_rn(sum, __shfl_sync(kFullMask, wv, j));
    if (lane < K) {
        topk_idx[(size_t)t * K + lane] = my_pick;
        topk_w[(size_t)t * K + lane] = __fdiv_rn(wv, sum);
    }
}

}  // namespace

cudaError_t launch_route(const float *logits, const float *bias, int T, int E, int K, int mode,
                         int n_group, int topk_group, int32_t *topk_idx, float *topk_w,
                         cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int grid = (T + kWarpsPerCta - 1) / kWarpsPerCta;
    const size_t smem = sizeof(float) * 2 * (size_t)E * kWarpsPerCta;
    if (mode == EP_ROUTE_SOFTMAX)
        route_kernel<EP_ROUTE_SOFTMAX><<<grid, kWarpsPerCta * 32, smem, stream>>>(
            logits, bias, T, E, K, n_group, topk_group, topk_idx, topk_w);
    else
        route_kernel<EP_ROUTE_GROUPED_SIGMOID><<<grid, kWarpsPerCta * 32, smem, stream>>>(
            logits, bias, T, E, K, n_group, topk_group, topk_idx, topk_w);
    return cudaGetLastError();
}

}  // namespace ep
