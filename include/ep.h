/*
 * ep.h -- MoE token dispatch and combine on one GPU (GB300, sm_103a): C ABI.
 *
 * The hot path of expert-parallel MoE layers, on one device whose HBM holds
 * every expert: logical expert-parallel ranks are only partitions of the
 * expert set.  Four operations:
 *
 *   ep_layout         top-k router output -> per-expert layout: expert
 *                     histogram, padded exclusive scan, stable slots.
 *   ep_dispatch       scatter token rows into that layout, optionally fused
 *                     with dynamic 1x128 FP8-E4M3 quantisation.
 *   ep_combine        top-k weighted reduction of expert outputs back to
 *                     token order.
 *   ep_masked_repack  contiguous expert segments -> masked [E, cap, H] slab.
 *
 * Sources (the pages describe a library integration, not kernels):
 *   [PR-24443]  SGLang PR "moe: add DeepEP V2 ElasticBuffer support to MoE
 *               token dispatcher", section "Motivation" (V2 dispatch infers
 *               the layout from topk_idx; per-expert receive counts live on
 *               the handle; combine reuses the dispatch handle) and the review
 *               thread on num_topk ("lots of kNumTopk <= 32 restrictions"),
 *               and its commit "num_max_tokens_per_rank sizing" (dispatch
 *               hard-asserts num_tokens <= num_max_tokens_per_rank).
 *   [PR-35634]  SGLang PR "[Feature] Add DeepEPv2 (ElasticBuffer) MoE A2A
 *               backend": "Supported scope" (decode uses the expanded masked
 *               layout, extend/prefill the contiguous layout; dynamic
 *               blockwise FP8), "Implementation" (masked-slab repack kernels;
 *               Hopper FP32 scales and Blackwell packed UE8M0 scales;
 *               single-use handles), "Capacity and fail-fast behavior".
 *   [DISC-26563] SGLang discussion "deepep v2 support?": the expert-format
 *               gate (128x128 blockwise FP8 with dynamic activation scaling,
 *               or unquantised BF16).
 *   [VLLM-EP]   vLLM tools/ep_kernels commit adding the deepep_v2 backend:
 *               do_expand=True gives a per-expert-contiguous layout, with
 *               weighted reduction in combine; FP8 block-quantised dispatch.
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     allocates no memory and never synchronises the host.  Its only state is
 *     a per-device cache of the SM count (read once with
 *     cudaDeviceGetAttribute) and, for ep_layout_noalloc alone, the fixed
 *     device array that call uses as scratch (with its looked-up address);
 *     every other entry point keeps nothing between calls.
 *   - Tracing: with the environment variable EP_NVTX=1 (read once per
 *     process) every entry point wraps its work in an NVTX range of its own
 *     name, for nsys / ncu timelines; off by default, and the ranges do
 *     nothing without a tool attached.
 *     Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and completes asynchronously.  Kernels are launched as
 *     programmatic dependents (programmatic dependent launch) and may start
 *     while the previous kernel on the stream finishes; each waits for it
 *     before touching its results, and the layout's first kernel before
 *     anything else.  Dispatch and combine let the next kernel start early:
 *     a caller's kernel launched as a programmatic dependent after them must
 *     itself wait (griddepcontrol.wait) before reading their outputs.
 *   - Host-detectable errors (bad shapes, NULL or misaligned pointers, too many
 *     tokens) are returned synchronously and nothing is launched.  A failed
 *     launch returns EP_ERR_CUDA.
 *   - Data-dependent errors are raised on the device into the layout's status
 *     word as the maximum of the codes seen (no trap, no assert, no
 *     out-of-bounds write): EP_ERR_BAD_EXPERT_ID for an id outside [-1, E),
 *     EP_ERR_CAPACITY for a masked expert receiving more than `capacity` rows,
 *     EP_ERR_TIMEOUT if a bulk copy a kernel waits for never completes (the
 *     wait is bounded; the kernel then waits, again for a bounded time, for
 *     the copies it issued and returns; if even that drain runs out, a copy
 *     may still be landing in a CTA that has exited, and the context should
 *     be treated as suspect).
 *     Read it back after the stream completes.
 *   - bf16 means IEEE binary32's upper 16 bits; FP8 means E4M3FN (OCP OFP8).
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ep_stream_t; /* identical to cudaStream_t */

typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,   /* bad shape, enum, NULL or misaligned pointer    */
    EP_ERR_CAPACITY = 2,      /* too many tokens / rows for the reserved space  */
    EP_ERR_BAD_EXPERT_ID = 3, /* device-side only: id outside [-1, E)          */
    EP_ERR_CUDA = 4,          /* a CUDA launch failed                           */
    EP_ERR_UNSUPPORTED = 5,   /* valid request this build does not implement    */
    EP_ERR_TIMEOUT = 6        /* device-side only: a bulk copy a kernel waited
                                 for did not complete within about a second    */
} ep_status_t;

typedef enum ep_layout_kind {
    EP_LAYOUT_CONTIG = 0, /* expanded per-expert-contiguous rows (prefill)  */
    EP_LAYOUT_MASKED = 1  /* [E, capacity, H] slab + per-expert counts (decode) */
} ep_layout_kind_t;

typedef enum ep_quant {
    EP_QUANT_NONE = 0,     /* bf16 rows                                           */
    EP_QUANT_FP8_F32 = 1,  /* E4M3 rows + fp32 scale per 1x128 group  [rows, H/128]  */
    EP_QUANT_FP8_UE8M0 = 2, /* E4M3 rows + UE8M0 exponent per group, 4 per int32 word
                              [rows, ceil(H/512)]                                   */
    EP_QUANT_MXFP8 = 3,     /* E4M3 rows + E8M0 scale per 1x32 block, 4 per int32 word
                              [rows, H/128] ([DISC-26563]: 1x32 MXFP8 with dynamic
                              activation scaling; OCP MX v1.0 conversion rule)       */
    EP_QUANT_FP8_UE8M0_MN = 4 /* as EP_QUANT_FP8_UE8M0, scale words stored MN-major for a
                              grouped GEMM's TMA: word p of every row contiguous along
                              the rows, columns padded to 4 rows (16 bytes):
                              contiguous [P][roundup(rows_capacity, 4)], masked
                              [E][P][roundup(capacity, 4)], P = ceil(H/512)
                              ([PR-35634] "Implementation": Blackwell packed UE8M0) */
} ep_quant_t;

typedef enum ep_route {
    EP_ROUTE_SOFTMAX = 0,        /* softmax top-K, weights renormalised over the picks */
    EP_ROUTE_GROUPED_SIGMOID = 1 /* sigmoid + bias, group-limited top-K (DeepSeek-V3)  */
} ep_route_t;

#define EP_MAX_HIDDEN 32768 /* largest hidden size H (shared-memory row staging) */
#define EP_MAX_TOPK 32     /* [PR-24443] review: kNumTopk <= 32 */
#define EP_MAX_EXPERTS 1024
#define EP_MAX_ALIGN 128

/*
 * The layout ("handle"): shape plus caller-owned device arrays.  ep_layout()
 * fills the arrays; ep_dispatch() and ep_combine() read them, so combine
 * reuses exactly the dispatch handle ([PR-24443] "Motivation"; [PR-35634]
 * "Implementation").  T = num_tokens, K = num_topk, E = num_experts.
 *
 * Row space: contiguous -> rows = expert_offset[E] (at most ep_rows_capacity);
 *            masked     -> rows = E * capacity, expert e owns rows
 *                          [e*capacity, (e+1)*capacity).
 */
typedef struct ep_layout {
    /* shape, set by the caller */
    int32_t num_tokens;  /* T >= 0                                                 */
    int32_t num_topk;    /* K in [1, EP_MAX_TOPK]                                   */
    int32_t num_experts; /* E in [1, EP_MAX_EXPERTS]                                */
    int32_t num_ranks;   /* R >= 1 logical ranks, R divides E; rank r owns experts
                            [r*E/R, (r+1)*E/R)                                      */
    int32_t kind;        /* ep_layout_kind_t                                        */
    int32_t align;       /* contiguous: segment alignment in rows, a power of two in
                            [1, EP_MAX_ALIGN]; masked: ignored                      */
    int32_t capacity;    /* masked: slots per expert, >= 1; contiguous: ignored      */
    int32_t max_tokens;  /* reserved token capacity: T > max_tokens is rejected with
                            EP_ERR_CAPACITY before any launch ([PR-24443] commit
                            "num_max_tokens_per_rank sizing"; [PR-35634] "Capacity
                            and fail-fast behavior").  0 = no limit.               */
    /* device arrays, caller-owned, int32 */
    int32_t *dst_row;       /* [T*K] row of entry (t,k) = t*K+k; -1 if not placed   */
    int32_t *row_src;       /* [rows] entry t*K+k that fills each row, -1 for padding
                               and empty slots; may be NULL                        */
    int32_t *expert_count;  /* [E] expert histogram (rows requested per expert)     */
    int32_t *expert_offset; /* [E+1] first row of each expert; [E] = rows            */
    int32_t *rank_rows;     /* [R] rows requested per logical rank; may be NULL       */
    int32_t *status;        /* [1] device status word, reset by ep_layout            */
} ep_layout_t;

/* Human-readable name of a status code (static storage). */
const char *ep_status_str(ep_status_t status);

/* Rows a row buffer / row_src must hold: contiguous T*K + min(E, T*K)*(align-1)
 * (the worst case of the padded scan), masked E*capacity.  -1 on a bad layout. */
int64_t ep_rows_capacity(const ep_layout_t *layout);

/* 32-bit scale words per row: H/128 (fp32 scales, or MXFP8's H/32 E8M0 bytes),
 * ceil(H/512) (packed UE8M0), 0 (bf16); -1 if `hidden` is not valid for `quant`. */
int64_t ep_scale_cols(int32_t hidden, ep_quant_t quant);

/* 32-bit words the scale buffer of `quant` needs for this layout's row space:
 * rows_capacity * ep_scale_cols for the row-major modes, the padded MN-major
 * size for EP_QUANT_FP8_UE8M0_MN, 0 for bf16; -1 on a bad layout or hidden. */
int64_t ep_scale_words(const ep_layout_t *layout, int32_t hidden, ep_quant_t quant);

/* Bytes of device scratch ep_layout() needs for this shape (may be 0).  The
 * scratch holds per-tile expert histograms between the two layout kernels. */
size_t ep_layout_workspace_bytes(const ep_layout_t *layout);

/*
 * ep_layout -- expert histogram, padded exclusive scan, stable slot assignment
 * ([PR-24443] "Motivation": V2 dispatch infers the layout from topk_idx and
 * returns the per-expert receive counts; [PR-35634] "Supported scope" /
 * [VLLM-EP]: per-expert-contiguous and masked layouts).
 *
 *   topk_idx   device int32 [T, K], row-major; -1 = not routed.
 *   layout     shape + output arrays (see ep_layout_t); status is reset to 0.
 *   workspace  device scratch of at least ep_layout_workspace_bytes() bytes
 *              (NULL allowed when that is 0), 4-byte aligned; clobbered.
 *
 * Computes, for every entry i = t*K+k with e = topk_idx[i] in [0, E):
 *   expert_count[e]  = #entries with id e
 *   expert_offset    = contiguous: exclusive scan of roundup(count, align);
 *                      masked: e*capacity
 *   slot(i)          = #entries j < i with the same id (ascending token, then k)
 *   dst_row[i]       = expert_offset[e] + slot(i); -1 for -1 ids, bad ids, and
 *                      masked slots >= capacity (EP_ERR_CAPACITY raised)
 *   row_src[dst_row[i]] = i; every other row of the row space = -1
 *   rank_rows[r]     = sum of expert_count over rank r's experts
 *
 * Up to 16384 entries (T*K) one kernel of thread-block clusters computes
 * the layout and no workspace is needed; a cluster has 16 CTAs where the
 * device can co-schedule them, else 8.  The environment variable
 * EP_MAX_CLUSTER_CTAS=8 (read once per process; any value below 16 counts
 * as 8) caps it at 8, for a device partition that cannot place 16
 * co-scheduled CTAs.  A cluster's CTAs
 * exchange their histograms by bulk copies between their shared memories;
 * should one never complete, the bounded wait raises EP_ERR_TIMEOUT and the
 * layout's arrays are not valid.
 */
ep_status_t ep_layout(const int32_t *topk_idx, const ep_layout_t *layout, void *workspace,
                      size_t workspace_bytes, ep_stream_t stream);

/*
 * ep_dispatch -- scatter token rows into the layout, fused with dynamic 1x128
 * FP8-E4M3 quantisation ([PR-35634] "Supported scope", "Implementation";
 * [DISC-26563] 128x128 blockwise FP8 with dynamic activation scaling;
 * [VLLM-EP] FP8 block-quantised dispatch).
 *
 *   x           device bf16 [T, hidden], 16-byte aligned.
 *   hidden      H in [1, EP_MAX_HIDDEN]; a multiple of 128 for FP8, of 8 for bf16.
 *   out_rows    device [rows, H]: bf16 (EP_QUANT_NONE) or E4M3 bytes; 16-byte
 *               aligned.  Only rows named by dst_row are written; padding rows
 *               and empty slots are left untouched.
 *   out_scales  device [rows, ep_scale_cols(H, quant)] fp32 or int32 (for
 *               EP_QUANT_FP8_UE8M0_MN: ep_scale_words() int32, MN-major), 4-byte
 *               aligned; NULL for EP_QUANT_NONE.
 *   topk_w      optional device fp32 [T, K]; with row_w (device fp32 [rows]),
 *               row_w[dst_row[i]] = topk_w[i]. Both NULL to skip.
 *
 * For each token t and 128-wide group g of x[t]:
 *   amax  = max |x|;  s = max(amax, 1e-4) / 448   (fp32, IEEE division)
 *   FP8_F32:   q = E4M3_rn_satfinite(x / s), scale = s
 *   FP8_UE8M0: s rounded up to 2^(e-127) (e = biased exponent of s, plus one
 *              when s is not a power of two); q = E4M3_rn_satfinite(x * 2^(127-e));
 *              byte g%4 of int32 word g/4 (little-endian) = e; unused bytes 127.
 *   MXFP8:     per 32-element block b: X = 2^(floor(log2 amax) - 8) (8 = exponent
 *              of E4M3's largest normal), clamped at 2^-127 (all-zero and
 *              subnormal blocks); q = E4M3_rn_satfinite(x / X) (values between
 *              448 and 512 saturate); byte b%4 of int32 word b/4 = log2(X) + 127.
 * and the same bytes are written to every row dst_row[t*K+k] >= 0.
 *
 * Ordering: the kernels are programmatic dependents of the previous work on
 * the stream.  Dispatch reads x before it waits for its predecessor (to
 * overlap the layout), so x must be complete when that predecessor started:
 * always the case directly after ep_layout (whose first kernel waits for all
 * earlier work); a kernel that writes x and triggers its dependents early
 * (griddepcontrol.launch_dependents) must not run directly before ep_dispatch.
 */
ep_status_t ep_dispatch(const ep_layout_t *layout, const void *x, int32_t hidden,
                        ep_quant_t quant, void *out_rows, void *out_scales,
                        const float *topk_w, float *row_w, ep_stream_t stream);

/*
 * ep_layout_dispatch -- ep_layout followed by ep_dispatch in one call: the
 * dispatch that "infers the layout from topk_idx" itself ([PR-24443]
 * "Motivation": V2 folds V1's separate dispatch-layout pre-pass into
 * dispatch).  Arguments, outputs and errors are exactly those of the two
 * calls (topk_idx, layout and workspace as for ep_layout; x, hidden, quant,
 * out_rows, out_scales, topk_w, row_w as for ep_dispatch), and the results
 * are bit-identical to them.  The two kernels are launched back to back, the
 * dispatch as a programmatic dependent of the layout (its first rows load
 * and quantise while the layout runs).
 */
ep_status_t ep_layout_dispatch(const int32_t *topk_idx, const ep_layout_t *layout,
                               void *workspace, size_t workspace_bytes, const void *x,
                               int32_t hidden, ep_quant_t quant, void *out_rows,
                               void *out_scales, const float *topk_w, float *row_w,
                               ep_stream_t stream);

/*
 * ep_selftest_bounded_wait -- diagnostic with no counterpart in the pages:
 * checks on this GPU that the bounded waits of the dispatch kernels give up
 * instead of hanging.  One CTA waits on a shared-memory barrier that expects
 * bytes no copy will deliver, for at most `limit_clocks` SM clocks
 * (1 .. 2^31), then raises EP_ERR_TIMEOUT into the device word *status
 * (caller-owned, 4-byte aligned; its previous value is kept if larger).
 */
ep_status_t ep_selftest_bounded_wait(int32_t *status, int64_t limit_clocks, ep_stream_t stream);

/*
 * ep_selftest_cluster_wait -- diagnostic with no counterpart in the pages:
 * the same check for the bounded wait of the decode layout's histogram
 * exchange.  Two CTAs of one thread-block cluster each wait for bytes no
 * peer sends, for at most `limit_clocks` SM clocks (1 .. 2^31), still meet
 * at the closing cluster barrier, and raise EP_ERR_TIMEOUT into *status
 * (caller-owned, 4-byte aligned; its previous value is kept if larger).
 */
ep_status_t ep_selftest_cluster_wait(int32_t *status, int64_t limit_clocks, ep_stream_t stream);

/*
 * ep_combine -- top-k weighted reduction back to token order ([VLLM-EP]
 * "weighted reduction in combine"; combine reuses the dispatch handle,
 * [PR-24443] "Motivation").  The reduction is applied exactly once.
 *
 *   y        device bf16 expert outputs in the layout's row space [rows, H]
 *            (masked: [E, capacity, H]), 16-byte aligned.
 *   topk_w   device fp32 [T, K].
 *   out      device bf16 [T, H], 16-byte aligned; every element is written.
 *
 *   out[t,h] = bf16_rn( sum over k = 0..K-1 with dst_row[t*K+k] >= 0 of
 *                       topk_w[t,k] * y[dst_row[t*K+k], h] )
 * accumulated in fp32 in ascending k, each product and sum rounded separately
 * (no fused multiply-add); a token with no placed entry gets +0.
 */
ep_status_t ep_combine(const ep_layout_t *layout, const void *y, int32_t hidden,
                       const float *topk_w, void *out, ep_stream_t stream);

/*
 * ep_masked_repack -- copy a contiguous layout's expert segments into the
 * masked decode slab ([PR-35634] "Implementation": masked-slab repack kernels
 * with Hopper FP32 and Blackwell packed UE8M0 scales).
 *
 *   layout       a CONTIGUOUS layout already filled by ep_layout().
 *   rows         device [rows, H] bf16 or E4M3 (as written by ep_dispatch).
 *   row_scales   device [rows, ep_scale_cols] or NULL for EP_QUANT_NONE
 *                (EP_QUANT_FP8_UE8M0_MN: the contiguous layout's MN-major words,
 *                and slab_scales receives the masked MN-major layout).
 *   capacity     slab slots per expert, >= 1.
 *   slab         device [E, capacity, H]; slab_scales [E, capacity, cols].
 *   masked_m     device int32 [E] = min(expert_count[e], capacity).
 *
 *   slab[e, s] = rows[expert_offset[e] + s] for s < masked_m[e]; other slab rows
 *   are untouched.  expert_count[e] > capacity raises EP_ERR_CAPACITY into the
 *   layout's status word.
 */
ep_status_t ep_masked_repack(const ep_layout_t *layout, const void *rows,
                             const void *row_scales, int32_t hidden, ep_quant_t quant,
                             int32_t capacity, void *slab, void *slab_scales,
                             int32_t *masked_m, ep_stream_t stream);

/*
 * ep_route_topk -- router output from logits: the topk_idx / topk_w that
 * ep_layout and ep_combine take ([PR-24443] "Motivation": V2 dispatch infers
 * its layout from topk_idx), for the router families of the models
 * [PR-35634] "Supported scope" lists (Qwen3-MoE softmax, DeepSeek-V3/V4
 * grouped sigmoid).
 *
 *   logits     device fp32 [T, E], finite.
 *   bias       device fp32 [E] added to the sigmoid scores (grouped mode), or
 *              NULL for none; ignored in softmax mode.
 *   mode       EP_ROUTE_SOFTMAX: the K largest softmax probabilities (the K
 *              largest logits), w = p / sum(p over the K).
 *              EP_ROUTE_GROUPED_SIGMOID: s = sigmoid(logit), c = s + bias;
 *              group score = sum of the two largest c in each of n_group
 *              groups of E/n_group; the topk_group best groups are kept; the
 *              K largest c among their experts; w = s / sum(s over the K).
 *   n_group, topk_group  grouped mode: 1 <= n_group <= 32, E % n_group == 0,
 *              E/n_group >= 2, 1 <= topk_group <= n_group,
 *              K <= topk_group * E / n_group; ignored in softmax mode.
 *   topk_idx   device int32 [T, K] (picks in rank order); topk_w fp32 [T, K].
 * Ties go to the lower expert / group id; selections are decided in fp32.
 */
ep_status_t ep_route_topk(const float *logits, const float *bias, int32_t num_tokens,
                          int32_t num_experts, int32_t num_topk, ep_route_t mode,
                          int32_t n_group, int32_t topk_group, int32_t *topk_idx, float *topk_w,
                          ep_stream_t stream);

/*
 * ep_rank_layout -- per-logical-rank deduplicated send layout: a token is sent
 * once to every logical rank owning one of its experts (the dispatch-layout
 * pre-pass [PR-24443] "Motivation" says V2 infers internally; [VLLM-EP]
 * intra/inter-node expert parallelism).  Rank r owns experts
 * [r*E/R, (r+1)*E/R).
 *
 *   topk_idx     device int32 [T, K] expert ids (E = num_experts).
 *   rank_idx     device int32 [T*K], written: the rank of entry (t,k) if no
 *                earlier k of token t named that rank, else -1 (-2 for ids
 *                outside [-1, E), reported as EP_ERR_BAD_EXPERT_ID).
 *   rank_layout  a contiguous ep_layout_t with num_experts = R (R divides E),
 *                num_tokens = T, num_topk = K, filled as ep_layout() fills it
 *                from rank_idx: dst_row[t*K+k] is the send row of (t, rank) at
 *                the entry that first names the rank, expert_count[r] the
 *                tokens sent to rank r, expert_offset the rank-major segments
 *                (ascending tokens inside a rank), row_src the entry per row.
 *   workspace    as for ep_layout() with rank_layout's shape.
 * ep_dispatch(rank_layout, ...) then writes each token once per rank.
 */
ep_status_t ep_rank_layout(const int32_t *topk_idx, int32_t num_experts, int32_t *rank_idx,
                           const ep_layout_t *rank_layout, void *workspace,
                           size_t workspace_bytes, ep_stream_t stream);

/*
 * ep_rank_expand -- the receiving side's local expand: row dst_row[t,k] of
 * `layout` (the per-expert layout of the same topk_idx) receives the send row
 * of (t, rank of topk_idx[t,k]), with its scale row.  quant is the mode the
 * send buffer was dispatched with; the MN-major scale layout is not
 * supported here (EP_ERR_UNSUPPORTED).  Rows dst_row < 0 are skipped.
 * expand(dispatch(rank_layout, x)) equals dispatch(layout, x) byte for byte.
 */
ep_status_t ep_rank_expand(const ep_layout_t *rank_layout, const ep_layout_t *layout,
                           const int32_t *topk_idx, int32_t hidden, ep_quant_t quant,
                           const void *send_rows, const void *send_scales, void *out_rows,
                           void *out_scales, ep_stream_t stream);

/*
 * ep_layout_noalloc -- ep_layout with its scratch taken from a fixed array
 * inside the library, for callers that cannot allocate device memory (a
 * serving runtime that reserves all memory at start-up and forbids later
 * allocation, a plugin handed only its input and output buffers, C code
 * without a device allocator).  The pages have no counterpart to this call.
 *
 *   Same arguments and results as ep_layout, minus the workspace.
 *   The array holds EP_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 *   library, until the process exits.  Arguments are checked first, exactly
 *   as ep_layout checks them (same codes); then a shape whose
 *   ep_layout_workspace_bytes() exceeds the array is rejected with
 *   EP_ERR_CAPACITY, still before any launch.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make it before any stream capture.  The address is kept
 *   per device and CUDA context: after cudaDeviceReset the next call looks it
 *   up again in the new context (again before any capture).  All calls share the
 *   array: calls whose work overlaps on the GPU race and must be ordered by
 *   the caller (one stream, or events).  Nothing in the array needs clearing
 *   between calls.
 */
#define EP_NOALLOC_SCRATCH_BYTES (256u * 1024u)
ep_status_t ep_layout_noalloc(const int32_t *topk_idx, const ep_layout_t *layout,
                              ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
