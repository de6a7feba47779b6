/*
 * CPU oracle for MoE token dispatch / combine -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct C.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it; the library never calls it.  It shares
 * no code, header, table or constant with the CUDA path.
 *
 * Every function follows one definition, stated beside it in oracle.c:
 *   - layout: expert histogram, padded exclusive scan, stable slot in
 *     ascending (token, k) order (the "infers layout from topk_idx" step of
 *     SGLang PR "add DeepEP V2 ElasticBuffer support to MoE token dispatcher",
 *     section "Motivation"; the contiguous / masked layouts of SGLang PR
 *     "Add DeepEPv2 (ElasticBuffer) MoE A2A backend", section "Supported scope");
 *   - dispatch: row scatter fused with dynamic 1x128 FP8-E4M3 quantisation with
 *     fp32 or packed UE8M0 scales (same PR, section "Implementation"; SGLang
 *     discussion "deepep v2 support?", the 128x128 blockwise FP8 gate), or
 *     1x32 MXFP8 (the same discussion's "1x32 MXFP8 ... with dynamic
 *     activation scaling", with the OCP Microscaling Formats (MX) v1.0
 *     conversion rule for the shared scale);
 *   - combine: top-k weighted reduction back to token order (vLLM
 *     tools/ep_kernels commit message, "weighted reduction in combine");
 *   - masked repack: contiguous expert segments -> [E, cap, H] slab;
 *   - router top-k before the layout (softmax top-K renormalised; DeepSeek-V3
 *     style grouped sigmoid with bias), the step whose output topk_idx V2
 *     dispatch takes (first SGLang PR, "Motivation"); no page gives its
 *     formulas, so it follows the model families the second PR's "Supported
 *     scope" names;
 *   - per-rank deduplicated send layout and local expand: each token sent once
 *     to every logical rank owning one of its experts (the V1 dispatch-layout
 *     pre-pass the first SGLang PR's "Motivation" says V2 folds into dispatch,
 *     and the vLLM commit's intra/inter-node expert parallelism).
 *
 * Parity pins: every function here is pinned by tests (brute force, closed
 * forms, library cross-checks) except two choices the pages leave open, whose
 * correctness is fixed only by their written definition ("parity unpinned"):
 * the 1e-4 clamp of amax before the scale is formed, and the byte order of
 * the packed UE8M0 words (byte g%4 of word g/4, little-endian, pad bytes 127).
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Oracle status values (their own numbering, mirrored by the tests). */
#define ORC_OK 0
#define ORC_CAPACITY 2
#define ORC_BAD_EXPERT_ID 3

/* Quantisation modes of orc_dispatch / orc_masked_repack. */
#define ORC_Q_NONE 0      /* bf16 rows */
#define ORC_Q_FP8_F32 1   /* E4M3 rows + fp32 scale per 1x128 group */
#define ORC_Q_FP8_UE8M0 2 /* E4M3 rows + one UE8M0 byte per group, 4 per int32 */
#define ORC_Q_MXFP8 3     /* E4M3 rows + one E8M0 byte per 32 elements (OCP MX) */

uint16_t orc_bf16_round(float f);
float orc_bf16_to_float(uint16_t b);
uint8_t orc_e4m3_encode(float v);
double orc_e4m3_decode(uint8_t code);

void orc_quant_group_f32(const uint16_t *x, int n, uint8_t *q, float *scale);
void orc_quant_group_ue8m0(const uint16_t *x, int n, uint8_t *q, uint8_t *exp_byte);
void orc_quant_block_mx(const uint16_t *x, int n, uint8_t *q, uint8_t *scale_byte);

int orc_layout(const int32_t *topk_idx, int T, int K, int E, int R, int masked,
               int align, int cap, int32_t *count, int32_t *offset,
               int32_t *dst_row, int32_t *row_src, int32_t *rank_rows);

void orc_dispatch(const uint16_t *x, int T, int K, int H, int quant,
                  const int32_t *dst_row, void *out_rows, void *out_scales,
                  const float *topk_w, float *row_w);

void orc_combine(const uint16_t *y, const float *topk_w, const int32_t *dst_row,
                 int T, int K, int H, uint16_t *out);

void orc_rank_ids(const int32_t *topk_idx, int T, int K, int E, int R, int32_t *rank_idx);
void orc_rank_expand(const int32_t *topk_idx, int T, int K, int E, int R,
                     const int32_t *send_dst, const int32_t *dst_row, int row_bytes,
                     int scale_bytes, const void *send_rows, const void *send_scales,
                     void *out_rows, void *out_scales);

#define ORC_ROUTE_SOFTMAX 0
#define ORC_ROUTE_GROUPED_SIGMOID 1
void orc_route_topk(const float *logits, const float *bias, int T, int E, int K, int mode,
                    int n_group, int topk_group, int32_t *topk_idx, double *topk_w,
                    float *sel_score);

void orc_scales_mn_major(const int32_t *row_major, int rows, int P, int masked, int E,
                         int cap, int32_t *out);

int orc_masked_repack(const void *rows, const void *row_scales, int H, int quant,
                      const int32_t *offset, const int32_t *count, int E, int cap,
                      void *slab, void *slab_scales, int32_t *masked_m);

#ifdef __cplusplus
}
#endif
#endif /* EP_ORACLE_H */
