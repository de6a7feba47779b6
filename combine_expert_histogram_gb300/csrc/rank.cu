// Per-logical-rank deduplicated sending: ep_rank_layout and ep_rank_expand.
//
// Expert-parallel dispatch sends a token once to every rank that owns one of
// its experts and lets the receiving rank expand it to its local experts (the
// dispatch-layout pre-pass of DeepEP V1 that, per SGLang PR "moe: add DeepEP
// V2 ElasticBuffer support to MoE token dispatcher", section "Motivation",
// V2 folds into dispatch).  On one GPU the ranks are expert ranges of one HBM;
// this is the layout a cross-GPU exchange would send, one contiguous segment
// per rank.
//   * rank_ids_kernel: one thread per entry (t,k) writes the rank of its
//     expert if no earlier k of the same token named that rank, else -1; the
//     ordinary layout kernels then run on these ids with R "experts", giving
//     one send row per (token, rank), ranks in order, tokens ascending;
//   * ep_dispatch on that layout fills the send buffer (each token once per
//     rank);
//   * rank_expand_kernel: one CTA per token copies, for each k, the send row
//     of (t, rank of its expert) into row dst_row[t,k] of the per-expert
//     layout, with its scale row, in 16-byte (rows) and 4-byte (scales) words.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    rank_ids_kernel(const int32_t *__restrict__ idx, int TK, int K, int E, int per,
                    int32_t *__restrict__ rank_idx) {
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= TK) return;
    const int k = i % K;
    const int e = __ldg(idx + i);
    int out;
    if (e == -1) {
        out = -1;
    } else if (e < -1 || e >= E) {
        out = -2;  // reported by the layout as a bad id
    } else {
        const int r = e / per;
        out = r;
        for (int j = i - k; j < i; ++j) {
            const int ej = __ldg(idx + j);
            if (ej >= 0 && ej < E && ej / per == r) {
                out = -1;
                break;
            }
        }
    }
    rank_idx[i] = out;
}

__global__ void __launch_bounds__(kThreads)
    rank_expand_kernel(const int32_t *__restrict__ idx, int K, int E, int per,
                       const int32_t *send_dst, const int32_t *dst_row, int row_bytes,
                       int scale_bytes, const uint8_t *send_rows, const uint8_t *send_scales,
                       uint8_t *__restrict__ out_rows, uint8_t *__restrict__ out_scales) {
    // the send buffer is the previous kernel's output (programmatic launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int t = blockIdx.x;
    __shared__ int s_src[EP_MAX_TOPK], s_dst[EP_MAX_TOPK];
    if (threadIdx.x < K) {
        const int k = threadIdx.x;
        const int e = __ldg(idx + (size_t)t * K + k);
        const int d = ld_dep(dst_row + (size_t)t * K + k);
        int src = -1;
        if (d >= 0 && e >= 0 && e < E) {
            const int r = e / per;
            for (int j = 0; j <= k; ++j) {
                const int ej = __ldg(idx + (size_t)t * K + j);
                if (ej >= 0 && ej < E && ej / per == r) {
                    src = ld_dep(send_dst + (size_t)t * K + j);
                    break;
                }
            }
        }
        s_src[k] = src;
        s_dst[k] = src >= 0 ? d : -1;
    }
    __syncthreads();
    const int chunks = row_bytes >> 4;
    for (int j = threadIdx.x; j < K * chunks; j += kThreads) {
        const int k = j / chunks, c = j - k * chunks;
        if (s_dst[k] < 0) continue;
        const uint4 v = ld_dep_v4(send_rows + (size_t)s_src[k] * row_bytes + 16 * c);
        st_v4(out_rows + (size_t)s_dst[k] * row_bytes + 16 * c, v);
    }
    const int words = scale_bytes >> 2;
    for (int j = threadIdx.x; j < K * words; j += kThreads) {
        const int k = j / words, c = j - k * words;
        if (s_dst[k] < 0) continue;
        reinterpret_cast<uint32_t *>(out_scales + (size_t)s_dst[k] * scale_bytes)[c] =
            (uint32_t)ld_dep(reinterpret_cast<const int32_t *>(send_scales + (size_t)s_src[k] * scale_bytes) + c);
    }
}

}  // namespace

cudaError_t launch_rank_ids(const int32_t *topk_idx, int T, int K, int E, int R,
                            int32_t *rank_idx, cudaStream_t stream) {
    const int TK = T * K;
    if (TK == 0) return cudaSuccess;
    rank_ids_kernel<<<(TK + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        topk_idx, TK, K, E, E / R, rank_idx);
    return cudaGetLastError();
}

cudaError_t launch_rank_expand(const ep_layout_t &RL, const ep_layout_t &L,
                               const int32_t *topk_idx, int row_bytes, int scale_bytes,
                               const void *send_rows, const void *send_scales, void *out_rows,
                               void *out_scales, cudaStream_t stream) {
    if (L.num_tokens == 0) return cudaSuccess;
    return launch_kernel(rank_expand_kernel, L.num_tokens, kThreads, 0, stream, true, topk_idx,
                         L.num_topk, L.num_experts, L.num_experts / RL.num_experts, RL.dst_row,
                         L.dst_row, row_bytes, scale_bytes,
                         static_cast<const uint8_t *>(send_rows),
                         static_cast<const uint8_t *>(send_scales),
                         static_cast<uint8_t *>(out_rows), static_cast<uint8_t *>(out_scales));
}

}  // namespace ep
