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
// One warp per token.  Common shapes (E = 32 * a power of two, n_group
// dividing 32) keep each lane's E/32 contiguous experts in registers, merge
// group top-2 values with xor-shuffles and make each pick two redux.sync
// reductions; other shapes stage the scores in shared memory, lane g scores
// group g, and each pick is a lane-local scan plus five xor-shuffle rounds.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kWarpsPerCta = 4;

// Small router grids (at most one CTA per SM) are launched as programmatic
// dependents and let the layout launch early; larger ones are launched
// plainly and let it launch when they end.  Measured in CUDA-graph loops of
// route + layout + dispatch + combine: 256 tokens (64 CTAs) 9.3 -> 8.7 us
// with the early launches, while 1024 tokens (256 CTAs) went from 39.5 to
// 40.7-42.7 us with either of them: a large grid resident early takes
// registers that the still-running previous kernel's later waves need.
// `early` is that choice; the wait comes first in both cases (without the
// programmatic launch it returns at once): the previous kernel may have
// produced the logits and may still read topk_idx / topk_w.
__device__ __forceinline__ void route_pdl_prologue(bool early) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
                 float *__restrict__ topk_w, bool early) {
    extern __shared__ float smem[];
    route_pdl_prologue(early);
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

// Order-preserving map of a float onto an unsigned key (larger float, larger key).
__device__ __forceinline__ unsigned ordered(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Register-resident router for E = 32 * VP experts (VP a power of two) and, in
// grouped mode, n_group dividing 32: lane l owns experts [l*VP, (l+1)*VP), a
// group spans 32 / n_group whole lanes.  Each argmax round is two warp
// reductions (redux.sync): the largest key, then the lowest expert id holding it.
template <int VP, int MODE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    route_reg_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T,
                     int K, int n_group, int topk_group, int32_t *__restrict__ topk_idx,
                     float *__restrict__ topk_w, bool early) {
    route_pdl_prologue(early);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kWarpsPerCta + warp;
    if (t >= T) return;  // whole warps
    constexpr int E = 32 * VP;
    const int base = lane * VP;
    const float *l = logits + (size_t)t * E + base;
    float v[VP], sg[VP];  // selection score, and the weight source (logit or sigmoid)
#pragma unroll
    for (int i = 0; i < VP; ++i) {
        const float x = __ldg(l + i);
        if (MODE == EP_ROUTE_SOFTMAX) {
            v[i] = x;
            sg[i] = x;
        } else {
            const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
            sg[i] = s;
            v[i] = __fadd_rn(s, bias ? __ldg(bias + base + i) : 0.0f);
        }
    }
    if (MODE == EP_ROUTE_GROUPED_SIGMOID) {
        // the two largest scores of this lane, merged over the group's lanes
        float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
        for (int i = 0; i < VP; ++i) {
            const float x = v[i];
            if (x > a1) {
                a2 = a1;
                a1 = x;
            } else if (x > a2) {
                a2 = x;
            }
        }
        const int lpg = 32 / n_group;  // lanes per group (a power of two)
        for (int off = 1; off < lpg; off <<= 1) {
            const float b1 = __shfl_xor_sync(kFullMask, a1, off);
            const float b2 = __shfl_xor_sync(kFullMask, a2, off);
            const float hi = fmaxf(a1, b1);
            a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
            a1 = hi;
        }
        const float gscore = __fadd_rn(a1, a2);
        const unsigned g = (unsigned)(lane / lpg);
        unsigned keep = 0;
        for (int j = 0; j < topk_group; ++j) {
            const bool open = !((keep >> g) & 1u);
            const unsigned key = open ? ordered(gscore) : 0u;
            const unsigned m = __reduce_max_sync(kFullMask, key);
            const unsigned win = __reduce_min_sync(kFullMask, open && key == m ? g : 0xffffffffu);
            keep |= 1u << win;
        }
        if (!((keep >> g) & 1u)) {
#pragma unroll
            for (int i = 0; i < VP; ++i) v[i] = -INFINITY;
        }
    }
    unsigned taken = 0;
    int my_pick = 0;
    float my_src = 0.0f;
    for (int j = 0; j < K; ++j) {
        float bv = -INFINITY, bs = 0.0f;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < VP; ++i) {  // first maximum = lowest id among equals
            if (!((taken >> i) & 1u) && (bi < 0 || v[i] > bv)) {
                bv = v[i];
                bs = sg[i];
                bi = i;
            }
        }
        const unsigned key = bi >= 0 ? ordered(bv) : 0u;
        const unsigned m = __reduce_max_sync(kFullMask, key);
        const unsigned win =
            __reduce_min_sync(kFullMask, bi >= 0 && key == m ? (unsigned)(base + bi) : 0xffffffffu);
        const int owner = (int)(win / VP);
        const float src = __shfl_sync(kFullMask, bs, owner);
        if (lane == owner) taken |= 1u << (win - (unsigned)base);
        if (lane == j) {
            my_pick = (int)win;
            my_src = src;
        }
    }
    float wv = 0.0f;
    if (MODE == EP_ROUTE_SOFTMAX) {
        const float top = __shfl_sync(kFullMask, my_src, 0);
        if (lane < K) wv = expf(__fadd_rn(my_src, -top));
    } else if (lane < K) {
        wv = my_src;
    }
    float sum = 0.0f;  // ascending j
    for (int j = 0; j < K; ++j) sum = __fadd_rn(sum, __shfl_sync(kFullMask, wv, j));
    if (lane < K) {
        topk_idx[(size_t)t * K + lane] = my_pick;
        topk_w[(size_t)t * K + lane] = __fdiv_rn(wv, sum);
    }
}

// Programmatic launch and early trigger for grids of at most one CTA per SM.
bool route_early(int grid) { return grid <= sm_count(); }

template <int MODE>
cudaError_t launch_reg(int VP, int grid, cudaStream_t stream, const float *logits,
                       const float *bias, int T, int K, int n_group, int topk_group,
                       int32_t *topk_idx, float *topk_w) {
    const int threads = kWarpsPerCta * 32;
#define EP_ROUTE_CASE(V)                                                                      \
    case V:                                                                                   \
        return launch_kernel(route_reg_kernel<V, MODE>, grid, threads, 0, stream,             \
                             route_early(grid), logits, bias, T, K, n_group, topk_group,     \
                             topk_idx, topk_w, route_early(grid));
    switch (VP) {
        EP_ROUTE_CASE(1)
        EP_ROUTE_CASE(2)
        EP_ROUTE_CASE(4)
        EP_ROUTE_CASE(8)
        EP_ROUTE_CASE(16)
        EP_ROUTE_CASE(32)
        default:
            return cudaErrorInvalidValue;
    }
#undef EP_ROUTE_CASE
}

}  // namespace

cudaError_t launch_route(const float *logits, const float *bias, int T, int E, int K, int mode,
                         int n_group, int topk_group, int32_t *topk_idx, float *topk_w,
                         cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int grid = (T + kWarpsPerCta - 1) / kWarpsPerCta;
    // register-resident path: E = 32 * (power of two), groups of whole lanes
    const bool pow2 = (E & (E - 1)) == 0;
    const bool groups_ok = mode == EP_ROUTE_SOFTMAX || (32 % n_group == 0);
    if (E >= 32 && pow2 && groups_ok) {
        if (mode == EP_ROUTE_SOFTMAX)
            return launch_reg<EP_ROUTE_SOFTMAX>(E / 32, grid, stream, logits, bias, T, K,
                                                n_group, topk_group, topk_idx, topk_w);
        return launch_reg<EP_ROUTE_GROUPED_SIGMOID>(E / 32, grid, stream, logits, bias, T, K,
                                                    n_group, topk_group, topk_idx, topk_w);
    }
    const size_t smem = sizeof(float) * 2 * (size_t)E * kWarpsPerCta;
    if (mode == EP_ROUTE_SOFTMAX)
        return launch_kernel(route_kernel<EP_ROUTE_SOFTMAX>, grid, kWarpsPerCta * 32, smem, stream,
                             route_early(grid), logits, bias, T, E, K, n_group, topk_group, topk_idx,
                             topk_w, route_early(grid));
    return launch_kernel(route_kernel<EP_ROUTE_GROUPED_SIGMOID>, grid, kWarpsPerCta * 32, smem,
                         stream, route_early(grid), logits, bias, T, E, K, n_group, topk_group,
                         topk_idx, topk_w, route_early(grid));
}

}  // namespace ep
