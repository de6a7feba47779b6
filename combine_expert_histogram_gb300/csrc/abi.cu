// C ABI of the dispatch / combine library (declared in include/ep.h):
// argument validation, sizing helpers and the launches.  Every host-detectable
// error returns before anything is enqueued.
#include <limits.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

#include "ep_common.cuh"

namespace ep {

bool trace_enabled() {
    static const bool on = [] {
        const char *v = getenv("EP_NVTX");
        return v != nullptr && atoi(v) != 0;
    }();
    return on;
}
TraceRange::TraceRange(const char *name) : on(trace_enabled()) {
    if (on) nvtxRangePushA(name);
}
TraceRange::~TraceRange() {
    if (on) nvtxRangePop();
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int64_t rows_capacity(const ep_layout_t &L) {
    const int64_t TK = (int64_t)L.num_tokens * L.num_topk;
    if (L.kind == EP_LAYOUT_MASKED) return (int64_t)L.num_experts * L.capacity;
    const int64_t used = TK < L.num_experts ? TK : L.num_experts;
    return TK + used * (L.align - 1);
}

// Shape checks (sizing helpers need nothing else).
ep_status_t check_shape(const ep_layout_t *L) {
    if (!L) return EP_ERR_INVALID_ARG;
    if (L->num_tokens < 0 || L->num_topk < 1 || L->num_topk > EP_MAX_TOPK) return EP_ERR_INVALID_ARG;
    if (L->num_experts < 1 || L->num_experts > EP_MAX_EXPERTS) return EP_ERR_INVALID_ARG;
    if (L->num_ranks < 1 || L->num_experts % L->num_ranks != 0) return EP_ERR_INVALID_ARG;
    if (L->kind == EP_LAYOUT_CONTIG) {
        if (!is_pow2(L->align) || L->align > EP_MAX_ALIGN) return EP_ERR_INVALID_ARG;
    } else if (L->kind == EP_LAYOUT_MASKED) {
        if (L->capacity < 1) return EP_ERR_INVALID_ARG;
    } else {
        return EP_ERR_INVALID_ARG;
    }
    if (L->max_tokens < 0) return EP_ERR_INVALID_ARG;
    if ((int64_t)L->num_tokens * L->num_topk > INT_MAX) return EP_ERR_INVALID_ARG;
    if (rows_capacity(*L) > INT_MAX) return EP_ERR_INVALID_ARG;
    return EP_OK;
}

// Shape and pointer checks shared by every entry point.
ep_status_t check_layout(const ep_layout_t *L) {
    const ep_status_t st = check_shape(L);
    if (st != EP_OK) return st;
    if (!L->dst_row || !L->expert_count || !L->expert_offset || !L->status) return EP_ERR_INVALID_ARG;
    if (!aligned(L->dst_row, 4) || !aligned(L->expert_count, 4) || !aligned(L->expert_offset, 4) ||
        !aligned(L->status, 4) || !aligned(L->row_src, 4) || !aligned(L->rank_rows, 4))
        return EP_ERR_INVALID_ARG;
    if (L->max_tokens > 0 && L->num_tokens > L->max_tokens) return EP_ERR_CAPACITY;
    return EP_OK;
}

ep_status_t check_hidden(int32_t H, ep_quant_t quant) {
    if (H <= 0 || H > EP_MAX_HIDDEN) return EP_ERR_INVALID_ARG;
    if (quant == EP_QUANT_NONE) return H % 8 == 0 ? EP_OK : EP_ERR_INVALID_ARG;
    if (quant == EP_QUANT_FP8_F32 || quant == EP_QUANT_FP8_UE8M0 || quant == EP_QUANT_MXFP8 ||
        quant == EP_QUANT_FP8_UE8M0_MN)
        return H % 128 == 0 ? EP_OK : EP_ERR_INVALID_ARG;
    return EP_ERR_INVALID_ARG;
}

ep_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

}  // namespace

ep_status_t check_layout_call(const int32_t *topk_idx, const ep_layout_t *L) {
    const ep_status_t st = check_layout(L);
    if (st != EP_OK) return st;
    if (L->num_tokens > 0 && (!topk_idx || !aligned(topk_idx, 4))) return EP_ERR_INVALID_ARG;
    if (layout_plan(*L).smem > 227 * 1024) return EP_ERR_UNSUPPORTED;  // more entries than one CTA can rank
    return EP_OK;
}

}  // namespace ep

using namespace ep;

extern "C" {

const char *ep_status_str(ep_status_t s) {
    switch (s) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG: bad shape, enum, NULL or misaligned pointer";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY: more tokens or rows than the reserved capacity";
        case EP_ERR_BAD_EXPERT_ID: return "EP_ERR_BAD_EXPERT_ID: expert id outside [-1, num_experts)";
        case EP_ERR_CUDA: return "EP_ERR_CUDA: a CUDA launch failed";
        case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
        case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT: a device-side copy did not complete in time";
    }
    return "unknown ep_status_t";
}

int64_t ep_rows_capacity(const ep_layout_t *L) {
    if (check_shape(L) != EP_OK) return -1;
    return rows_capacity(*L);
}

int64_t ep_scale_cols(int32_t hidden, ep_quant_t quant) {
    if (check_hidden(hidden, quant) != EP_OK) return -1;
    if (quant == EP_QUANT_FP8_F32 || quant == EP_QUANT_MXFP8) return hidden / 128;
    if (quant == EP_QUANT_FP8_UE8M0 || quant == EP_QUANT_FP8_UE8M0_MN) return (hidden / 128 + 3) / 4;
    return 0;
}

int64_t ep_scale_words(const ep_layout_t *L, int32_t hidden, ep_quant_t quant) {
    if (check_shape(L) != EP_OK || check_hidden(hidden, quant) != EP_OK) return -1;
    const int64_t cols = ep_scale_cols(hidden, quant);
    if (quant != EP_QUANT_FP8_UE8M0_MN) return rows_capacity(*L) * cols;
    if (L->kind == EP_LAYOUT_MASKED)
        return (int64_t)L->num_experts * cols * ((L->capacity + 3) / 4 * 4);
    return cols * ((rows_capacity(*L) + 3) / 4 * 4);
}

size_t ep_layout_workspace_bytes(const ep_layout_t *L) {
    if (check_shape(L) != EP_OK) return 0;
    return layout_plan(*L).ws_bytes;
}

ep_status_t ep_layout(const int32_t *topk_idx, const ep_layout_t *L, void *workspace,
                      size_t workspace_bytes, ep_stream_t stream) {
    const TraceRange trace("ep_layout");
    const ep_status_t st = check_layout_call(topk_idx, L);
    if (st != EP_OK) return st;
    const LayoutPlan plan = layout_plan(*L);
    const size_t need = plan.ws_bytes;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 4)))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_layout(topk_idx, *L, static_cast<int32_t *>(workspace),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_dispatch(const ep_layout_t *L, const void *x, int32_t hidden, ep_quant_t quant,
                        void *out_rows, void *out_scales, const float *topk_w, float *row_w,
                        ep_stream_t stream) {
    const TraceRange trace("ep_dispatch");
    ep_status_t st = check_layout(L);
    if (st != EP_OK) return st;
    st = check_hidden(hidden, quant);
    if (st != EP_OK) return st;
    if (L->num_tokens == 0) return EP_OK;  // nothing to move
    if ((topk_w == nullptr) != (row_w == nullptr)) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_w, 4) || !aligned(row_w, 4)) return EP_ERR_INVALID_ARG;
    if (quant != EP_QUANT_NONE && (!out_scales || !aligned(out_scales, 4))) return EP_ERR_INVALID_ARG;
    if (!x || !out_rows || !aligned(x, 16) || !aligned(out_rows, 16)) return EP_ERR_INVALID_ARG;
    return from_cuda(launch_dispatch(*L, x, hidden, quant, out_rows, out_scales, topk_w, row_w,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_layout_dispatch(const int32_t *topk_idx, const ep_layout_t *L, void *workspace,
                               size_t workspace_bytes, const void *x, int32_t hidden,
                               ep_quant_t quant, void *out_rows, void *out_scales,
                               const float *topk_w, float *row_w, ep_stream_t stream) {
    const TraceRange trace("ep_layout_dispatch");
    // the argument rules of ep_layout and of ep_dispatch together
    ep_status_t st = check_layout(L);
    if (st != EP_OK) return st;
    if (L->num_tokens > 0 && (!topk_idx || !aligned(topk_idx, 4))) return EP_ERR_INVALID_ARG;
    const LayoutPlan plan = layout_plan(*L);
    if (plan.smem > 227 * 1024) return EP_ERR_UNSUPPORTED;
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 4)))
        return EP_ERR_INVALID_ARG;
    st = check_hidden(hidden, quant);
    if (st != EP_OK) return st;
    if (L->num_tokens > 0) {
        if ((topk_w == nullptr) != (row_w == nullptr)) return EP_ERR_INVALID_ARG;
        if (!aligned(topk_w, 4) || !aligned(row_w, 4)) return EP_ERR_INVALID_ARG;
        if (quant != EP_QUANT_NONE && (!out_scales || !aligned(out_scales, 4))) return EP_ERR_INVALID_ARG;
        if (!x || !out_rows || !aligned(x, 16) || !aligned(out_rows, 16)) return EP_ERR_INVALID_ARG;
    }
    return from_cuda(launch_layout_dispatch(topk_idx, *L, static_cast<int32_t *>(workspace), x,
                                            hidden, quant, out_rows, out_scales, topk_w, row_w,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_selftest_bounded_wait(int32_t *status, int64_t limit_clocks, ep_stream_t stream) {
    const TraceRange trace("ep_selftest_bounded_wait");
    if (!status || !aligned(status, 4) || limit_clocks < 1 || limit_clocks > (int64_t)1 << 31)
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_wait_selftest(status, (long long)limit_clocks,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_selftest_cluster_wait(int32_t *status, int64_t limit_clocks, ep_stream_t stream) {
    const TraceRange trace("ep_selftest_cluster_wait");
    if (!status || !aligned(status, 4) || limit_clocks < 1 || limit_clocks > (int64_t)1 << 31)
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_cluster_wait_selftest(status, (long long)limit_clocks,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_combine(const ep_layout_t *L, const void *y, int32_t hidden, const float *topk_w,
                       void *out, ep_stream_t stream) {
    const TraceRange trace("ep_combine");
    ep_status_t st = check_layout(L);
    if (st != EP_OK) return st;
    st = check_hidden(hidden, EP_QUANT_NONE);
    if (st != EP_OK) return st;
    if (L->num_tokens == 0) return EP_OK;
    if (!y || !topk_w || !out || !aligned(y, 16) || !aligned(out, 16) || !aligned(topk_w, 4))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_combine(*L, y, hidden, topk_w, out,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_masked_repack(const ep_layout_t *L, const void *rows, const void *row_scales,
                             int32_t hidden, ep_quant_t quant, int32_t capacity, void *slab,
                             void *slab_scales, int32_t *masked_m, ep_stream_t stream) {
    const TraceRange trace("ep_masked_repack");
    ep_status_t st = check_layout(L);
    if (st != EP_OK) return st;
    if (L->kind != EP_LAYOUT_CONTIG) return EP_ERR_INVALID_ARG;
    st = check_hidden(hidden, quant);
    if (st != EP_OK) return st;
    if (capacity < 1 || (int64_t)L->num_experts * capacity > INT_MAX) return EP_ERR_INVALID_ARG;
    if (!rows || !slab || !masked_m || !aligned(rows, 16) || !aligned(slab, 16) || !aligned(masked_m, 4))
        return EP_ERR_INVALID_ARG;
    if (quant != EP_QUANT_NONE &&
        (!row_scales || !slab_scales || !aligned(row_scales, 4) || !aligned(slab_scales, 4)))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_masked_repack(*L, rows, row_scales, hidden, quant, capacity, slab,
                                          slab_scales, masked_m,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_route_topk(const float *logits, const float *bias, int32_t T, int32_t E,
                          int32_t K, ep_route_t mode, int32_t n_group, int32_t topk_group,
                          int32_t *topk_idx, float *topk_w, ep_stream_t stream) {
    const TraceRange trace("ep_route_topk");
    if (T < 0 || E < 1 || E > EP_MAX_EXPERTS || K < 1 || K > EP_MAX_TOPK || K > E)
        return EP_ERR_INVALID_ARG;
    if (mode == EP_ROUTE_GROUPED_SIGMOID) {
        if (n_group < 1 || n_group > 32 || E % n_group != 0 || E / n_group < 2 ||
            topk_group < 1 || topk_group > n_group || K > topk_group * (E / n_group))
            return EP_ERR_INVALID_ARG;
    } else if (mode != EP_ROUTE_SOFTMAX) {
        return EP_ERR_INVALID_ARG;
    }
    if ((int64_t)T * E > INT_MAX) return EP_ERR_INVALID_ARG;
    if (T == 0) return EP_OK;
    if (!logits || !topk_idx || !topk_w || !aligned(logits, 4) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4) || !aligned(bias, 4))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_route(logits, mode == EP_ROUTE_GROUPED_SIGMOID ? bias : nullptr, T, E,
                                  K, (int)mode, n_group, topk_group, topk_idx, topk_w,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_rank_layout(const int32_t *topk_idx, int32_t num_experts, int32_t *rank_idx,
                           const ep_layout_t *RL, void *workspace, size_t workspace_bytes,
                           ep_stream_t stream) {
    const TraceRange trace("ep_rank_layout");
    ep_status_t st = check_layout(RL);
    if (st != EP_OK) return st;
    if (RL->kind != EP_LAYOUT_CONTIG) return EP_ERR_INVALID_ARG;
    if (num_experts < RL->num_experts || num_experts > EP_MAX_EXPERTS ||
        num_experts % RL->num_experts != 0)
        return EP_ERR_INVALID_ARG;
    const int TK = RL->num_tokens * RL->num_topk;
    if (TK > 0 && (!topk_idx || !rank_idx || !aligned(topk_idx, 4) || !aligned(rank_idx, 4)))
        return EP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = launch_rank_ids(topk_idx, RL->num_tokens, RL->num_topk, num_experts,
                                      RL->num_experts, rank_idx, s);
    if (err != cudaSuccess) return EP_ERR_CUDA;
    return ep_layout(rank_idx, RL, workspace, workspace_bytes, stream);
}

ep_status_t ep_rank_expand(const ep_layout_t *RL, const ep_layout_t *L, const int32_t *topk_idx,
                           int32_t hidden, ep_quant_t quant, const void *send_rows,
                           const void *send_scales, void *out_rows, void *out_scales,
                           ep_stream_t stream) {
    const TraceRange trace("ep_rank_expand");
    ep_status_t st = check_layout(RL);
    if (st != EP_OK) return st;
    st = check_layout(L);
    if (st != EP_OK) return st;
    st = check_hidden(hidden, quant);
    if (st != EP_OK) return st;
    if (quant == EP_QUANT_FP8_UE8M0_MN) return EP_ERR_UNSUPPORTED;  // row-major scales only
    if (RL->num_tokens != L->num_tokens || RL->num_topk != L->num_topk ||
        L->num_experts % RL->num_experts != 0)
        return EP_ERR_INVALID_ARG;
    if (L->num_tokens == 0) return EP_OK;
    if (!topk_idx || !send_rows || !out_rows || !aligned(send_rows, 16) || !aligned(out_rows, 16))
        return EP_ERR_INVALID_ARG;
    const int G = hidden / 128;
    const int row_bytes = quant == EP_QUANT_NONE ? 2 * hidden : hidden;
    const int scale_bytes = (quant == EP_QUANT_FP8_F32 || quant == EP_QUANT_MXFP8) ? 4 * G
                            : quant == EP_QUANT_FP8_UE8M0 ? 4 * ((G + 3) / 4) : 0;
    if (scale_bytes && (!send_scales || !out_scales || !aligned(send_scales, 4) ||
                        !aligned(out_scales, 4)))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_rank_expand(*RL, *L, topk_idx, row_bytes, scale_bytes, send_rows,
                                        send_scales, out_rows, out_scales,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
