/*
 * CPU oracle for MoE token dispatch / combine -- TEST INFRASTRUCTURE ONLY.
 * See oracle.h for scope.  Built with -ffp-contract=off so that every fp32
 * multiply and add below is a separately rounded IEEE operation.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 = the upper 16 bits of an IEEE binary32. */
float orc_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round binary32 -> bf16, to nearest, ties to even.  Within one sign, binary32
 * bit patterns are ordered like their magnitudes, so the two bf16 neighbours of
 * f are its truncation `lo` and the next pattern up; the low 16 bits are the
 * distance from `lo` in units of 2^-16 bf16 ulp.  Overflow rounds to inf. */
uint16_t orc_bf16_round(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lo = u & 0xFFFF0000u;
    uint32_t rem = u & 0x0000FFFFu;
    int round_up = rem > 0x8000u || (rem == 0x8000u && ((lo >> 16) & 1u));
    if (round_up) lo += 0x00010000u;
    return (uint16_t)(lo >> 16);
}

/* ------------------------------------------------------------ FP8 E4M3FN */

/* E4M3FN (OCP 8-bit floating point): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits.  No infinities; S.1111.111 is NaN; the largest finite
 * magnitude is 2^8 * 1.75 = 448 (code 0x7E).  Exponent field 0 holds the
 * subnormals m * 2^-9, m = 0..7. */
double orc_e4m3_decode(uint8_t code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
    if (e == 0xF && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Encode with round-to-nearest-even and saturation to +-448 ("satfinite").
 * The sign is kept for values that round to zero. NaN -> 0x7F. */
uint8_t orc_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range, step 2^-9; the product is exact and nearbyint
         * rounds half to even in the default rounding mode.  m == 8 is the
         * smallest normal 2^-6, whose code is also 8. */
        double m = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int ex;
    double f = frexp(a, &ex);        /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                  /* a = (2f) * 2^e, 2f in [1, 2), e in [-6, 8] */
    double m = nearbyint((2.0 * f - 1.0) * 8.0); /* exact scaling, then RNE */
    if (m == 8.0) {                  /* mantissa carried into the exponent */
        m = 0.0;
        e += 1;
    }
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)m));
}

/* ------------------------------------------------- 1x128 dynamic FP8 quant */

static float group_amax(const uint16_t *x, int n) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float v = fabsf(orc_bf16_to_float(x[i]));
        if (v > amax) amax = v;
    }
    return amax;
}

/* FP32-scale ("Hopper") format: scale = max(amax, 1e-4) / 448, q = E4M3(x / scale),
 * both fp32 divides correctly rounded. */
void orc_quant_group_f32(const uint16_t *x, int n, uint8_t *q, float *scale) {
    float s = fmaxf(group_amax(x, n), 1e-4f) / 448.0f;
    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) / s);
    *scale = s;
}

/* Packed UE8M0 ("Blackwell") format: the fp32 scale above rounded UP to a power
 * of two 2^(e-127), e = biased exponent of s plus one when s has a non-zero
 * mantissa; q = E4M3(x * 2^(127-e)) (a multiply by a power of two); the byte
 * stored is e. */
void orc_quant_group_ue8m0(const uint16_t *x, int n, uint8_t *q, uint8_t *exp_byte) {
    float s = fmaxf(group_amax(x, n), 1e-4f) / 448.0f;
    uint32_t bits;
    memcpy(&bits, &s, sizeof bits);
    int e = (int)((bits >> 23) & 0xFFu) + ((bits & 0x007FFFFFu) != 0u);
    float inv = ldexpf(1.0f, 127 - e);
    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) * inv);
    *exp_byte = (uint8_t)e;
}

/* MXFP8 (OCP Microscaling Formats (MX) v1.0, "conversion from a vector of
 * scalars"): one shared scale per block of 32 elements, X = 2^(floor(log2
 * amax) - 8), 8 being the exponent of E4M3's largest normal (448 = 1.75*2^8);
 * elements q = E4M3_rne_satfinite(x / X).  X is stored as an E8M0 byte (bias
 * 127) and clamped at its smallest value 2^-127 (byte 0), which also covers
 * all-zero and subnormal blocks.  For a normal amax, floor(log2 amax) is its
 * unbiased exponent, so the byte is max(0, biased_exponent(amax) - 8), and
 * x / X = x * 2^(127 - byte) is a multiply by a power of two. */
void orc_quant_block_mx(const uint16_t *x, int n, uint8_t *q, uint8_t *scale_byte) {
    float amax = group_amax(x, n);
    int e = 0; /* biased exponent of amax; 0 for zero and subnormals */
    if (amax >= ldexpf(1.0f, -126)) {
        int ex;
        frexpf(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
        e = ex - 1 + 127;
    }
    int byte = e - 8 > 0 ? e - 8 : 0;
    float inv = ldexpf(1.0f, 127 - byte);
    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) * inv);
    *scale_byte = (uint8_t)byte;
}

/* ---------------------------------------------------------------- layout */

static int round_up(int v, int a) { return (v + a - 1) / a * a; }

/* Expert histogram, padded exclusive scan, stable slot assignment.
 *
 *   count[e]   = #{(t,k) : topk_idx[t,k] == e}                  (-1 skipped)
 *   contig:  offset[0] = 0, offset[e+1] = offset[e] + roundup(count[e], align)
 *   masked:  offset[e] = e * cap
 *   slot(t,k)  = #{(t',k') <lex (t,k) : topk_idx[t',k'] == topk_idx[t,k]}
 *   dst_row[t*K+k] = offset[e] + slot, -1 for -1 ids, bad ids, or (masked)
 *                    slot >= cap;  row_src[dst_row[t*K+k]] = t*K+k, all other
 *                    rows of [0, rows) are -1 (rows = offset[E], or E*cap).
 *   rank_rows[r] = sum of count[e] over the experts of logical rank r, which
 *                  owns experts [r*E/R, (r+1)*E/R).
 * Ids outside [-1, E) are reported as ORC_BAD_EXPERT_ID and get no slot;
 * masked overflow is reported as ORC_CAPACITY; the larger code wins.
 * Visiting (t,k) in lexicographic order with one running counter per expert
 * gives exactly the slot defined above. */
int orc_layout(const int32_t *topk_idx, int T, int K, int E, int R, int masked,
               int align, int cap, int32_t *count, int32_t *offset,
               int32_t *dst_row, int32_t *row_src, int32_t *rank_rows) {
    int status = ORC_OK;
    for (int e = 0; e < E; ++e) count[e] = 0;
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) {
                if (status < ORC_BAD_EXPERT_ID) status = ORC_BAD_EXPERT_ID;
                continue;
            }
            count[e] += 1;
        }
    }
    offset[0] = 0;
    for (int e = 0; e < E; ++e)
        offset[e + 1] = masked ? (e + 1) * cap : offset[e] + round_up(count[e], align);

    int rows = offset[E];
    if (row_src)
        for (int r = 0; r < rows; ++r) row_src[r] = -1;

    int32_t *running = (int32_t *)calloc((size_t)(E > 0 ? E : 1), sizeof(int32_t));
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int i = t * K + k;
            int e = topk_idx[i];
            dst_row[i] = -1;
            if (e < 0 || e >= E) continue;
            int slot = running[e]++;
            if (masked && slot >= cap) {
                if (status < ORC_CAPACITY) status = ORC_CAPACITY;
                continue;
            }
            int dst = offset[e] + slot;
            dst_row[i] = dst;
            if (row_src) row_src[dst] = i;
        }
    }
    free(running);

    if (rank_rows) {
        int per = E / R;
        for (int r = 0; r < R; ++r) {
            int32_t s = 0;
            for (int e = r * per; e < (r + 1) * per; ++e) s += count[e];
            rank_rows[r] = s;
        }
    }
    return status;
}

/* -------------------------------------------------------------- dispatch */

/* For every token t and every k with dst_row[t*K+k] >= 0, write token t's row
 * to row dst_row[t*K+k] of out_rows:
 *   ORC_Q_NONE:      the bf16 row as is; out_scales unused.
 *   ORC_Q_FP8_F32:   E4M3 bytes [rows, H]; fp32 scales [rows, H/128].
 *   ORC_Q_FP8_UE8M0: E4M3 bytes [rows, H]; scale bytes [rows, 4*ceil(G/4)],
 *                    byte g = exponent of group g (byte g%4 of little-endian
 *                    int32 word g/4), unused trailing bytes = 127 (2^0).
 *   ORC_Q_MXFP8:     E4M3 bytes [rows, H]; E8M0 bytes [rows, H/32], byte b =
 *                    scale of elements 32b..32b+31 (H/128 int32 words).
 * row_w[dst] = topk_w[t*K+k] when both are given. */
void orc_dispatch(const uint16_t *x, int T, int K, int H, int quant,
                  const int32_t *dst_row, void *out_rows, void *out_scales,
                  const float *topk_w, float *row_w) {
    int G = H / 128;
    int P = (G + 3) / 4;
    uint8_t *q = (uint8_t *)malloc((size_t)(H > 0 ? H : 1));
    float *sc = (float *)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
    uint8_t *eb = (uint8_t *)malloc((size_t)(4 * P > 0 ? 4 * P : 1));
    uint8_t *mx = (uint8_t *)malloc((size_t)(H / 32 > 0 ? H / 32 : 1));
    for (int t = 0; t < T; ++t) {
        const uint16_t *xr = x + (size_t)t * H;
        if (quant == ORC_Q_FP8_F32) {
            for (int g = 0; g < G; ++g) orc_quant_group_f32(xr + g * 128, 128, q + g * 128, &sc[g]);
        } else if (quant == ORC_Q_FP8_UE8M0) {
            for (int b = 0; b < 4 * P; ++b) eb[b] = 127;
            for (int g = 0; g < G; ++g) orc_quant_group_ue8m0(xr + g * 128, 128, q + g * 128, &eb[g]);
        } else if (quant == ORC_Q_MXFP8) {
            for (int b = 0; b < H / 32; ++b) orc_quant_block_mx(xr + b * 32, 32, q + b * 32, &mx[b]);
        }
        for (int k = 0; k < K; ++k) {
            int dst = dst_row[t * K + k];
            if (dst < 0) continue;
            if (quant == ORC_Q_NONE) {
                memcpy((uint16_t *)out_rows + (size_t)dst * H, xr, sizeof(uint16_t) * (size_t)H);
            } else {
                memcpy((uint8_t *)out_rows + (size_t)dst * H, q, (size_t)H);
                if (quant == ORC_Q_FP8_F32)
                    memcpy((float *)out_scales + (size_t)dst * G, sc, sizeof(float) * (size_t)G);
                else if (quant == ORC_Q_FP8_UE8M0)
                    memcpy((uint8_t *)out_scales + (size_t)dst * 4 * P, eb, (size_t)(4 * P));
                else
                    memcpy((uint8_t *)out_scales + (size_t)dst * (H / 32), mx, (size_t)(H / 32));
            }
            if (topk_w && row_w) row_w[dst] = topk_w[t * K + k];
        }
    }
    free(q);
    free(sc);
    free(eb);
    free(mx);
}

/* --------------------------------------------------------------- combine */

/* out[t, h] = bf16_rne( sum_{k ascending, dst_row[t*K+k] >= 0} w[t,k] * y[dst, h] )
 * accumulated in fp32 from 0.0f, each product and each sum rounded on its own.
 * A token with no routed expert gets +0. */
void orc_combine(const uint16_t *y, const float *topk_w, const int32_t *dst_row,
                 int T, int K, int H, uint16_t *out) {
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int dst = dst_row[t * K + k];
                if (dst < 0) continue;
                float p = topk_w[t * K + k] * orc_bf16_to_float(y[(size_t)dst * H + h]);
                acc = acc + p;
            }
            out[(size_t)t * H + h] = orc_bf16_round(acc);
        }
    }
}

/* ------------------------------------------------------------ router top-k */

/* Is (va, a) ranked before (vb, b)?  Larger value first, lower index on ties. */
static int ranks_before(double va, int a, double vb, int b) { return va > vb || (va == vb && a < b); }

/* Top-K selection by repeated maximum over `score` (entries with keep[e] == 0
 * are excluded); writes the chosen indices in rank order. */
static void select_top(const double *score, const int *keep, int n, int k, int *out) {
    int *taken = (int *)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < n; ++e) {
            if (taken[e] || (keep && !keep[e])) continue;
            if (best < 0 || ranks_before(score[e], e, score[best], best)) best = e;
        }
        out[j] = best;
        if (best >= 0) taken[best] = 1;
    }
    free(taken);
}

/* Router output for T tokens of E logits.
 *   SOFTMAX: p = softmax(logits); topk_idx = the K largest p (ties to the lower
 *     expert id; p is monotone in the logit, so the logits decide);
 *     topk_w = p_sel / sum(p_sel).
 *   GROUPED_SIGMOID (DeepSeek-V3 style): s = sigmoid(logit), c = s + bias, the
 *     selection score, computed in fp32 (the precision the decision is taken
 *     in); experts split into n_group groups of E/n_group; group score = sum
 *     of its two largest c; the topk_group best groups are kept (ties to the
 *     lower group id); topk_idx = the K largest c among kept experts;
 *     topk_w = s_sel / sum(s_sel).
 * Weights are computed in fp64.  sel_score[t*K+j] is the fp32 selection score
 * of the j-th pick (logit, or c), for tie analysis in tests. */
void orc_route_topk(const float *logits, const float *bias, int T, int E, int K, int mode,
                    int n_group, int topk_group, int32_t *topk_idx, double *topk_w,
                    float *sel_score) {
    double *score = (double *)malloc(sizeof(double) * (size_t)E);
    double *sig = (double *)malloc(sizeof(double) * (size_t)E);
    float *c32 = (float *)malloc(sizeof(float) * (size_t)E);
    int *keep = (int *)malloc(sizeof(int) * (size_t)E);
    int *pick = (int *)malloc(sizeof(int) * (size_t)(K > 0 ? K : 1));
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        if (mode == ORC_ROUTE_SOFTMAX) {
            double m = -INFINITY, z = 0.0;
            for (int e = 0; e < E; ++e) m = l[e] > m ? l[e] : m;
            for (int e = 0; e < E; ++e) {
                sig[e] = exp((double)l[e] - m);  /* unnormalised softmax */
                z += sig[e];
                score[e] = l[e];
            }
            for (int e = 0; e < E; ++e) sig[e] /= z;
            select_top(score, NULL, E, K, pick);
        } else {
            int gs = E / n_group;
            for (int e = 0; e < E; ++e) {
                float s32 = 1.0f / (1.0f + expf(-l[e]));
                c32[e] = s32 + (bias ? bias[e] : 0.0f);
                sig[e] = 1.0 / (1.0 + exp(-(double)l[e]));
                score[e] = c32[e];
            }
            double *gscore = (double *)malloc(sizeof(double) * (size_t)n_group);
            int *gpick = (int *)malloc(sizeof(int) * (size_t)n_group);
            for (int g = 0; g < n_group; ++g) {
                int two[2];
                select_top(score + (size_t)g * gs, NULL, gs, 2, two);
                gscore[g] = (double)((float)score[g * gs + two[0]] + (float)score[g * gs + two[1]]);
            }
            select_top(gscore, NULL, n_group, topk_group, gpick);
            for (int e = 0; e < E; ++e) keep[e] = 0;
            for (int j = 0; j < topk_group; ++j)
                for (int e = gpick[j] * gs; e < (gpick[j] + 1) * gs; ++e) keep[e] = 1;
            select_top(score, keep, E, K, pick);
            free(gscore);
            free(gpick);
        }
        double sum = 0.0;
        for (int j = 0; j < K; ++j) sum += sig[pick[j]];
        for (int j = 0; j < K; ++j) {
            topk_idx[t * K + j] = pick[j];
            topk_w[t * K + j] = sig[pick[j]] / sum;
            if (sel_score) sel_score[t * K + j] = (float)score[pick[j]];
        }
    }
    free(score);
    free(sig);
    free(c32);
    free(keep);
    free(pick);
}

/* ------------------------------------------ per-rank deduplicated sending */

/* Logical rank r owns experts [r*E/R, (r+1)*E/R).  rank_idx[t*K+k] is the rank
 * of expert topk_idx[t,k] the first time token t names that rank (ascending
 * k), -1 for later entries of the same rank and for -1 ids; ids outside
 * [-1, E) become -2 so that the layout over ranks reports them.  Running
 * orc_layout on rank_idx with R "experts" then gives the rank-major send
 * layout: one row per (token, rank) pair, ascending tokens inside a rank. */
void orc_rank_ids(const int32_t *topk_idx, int T, int K, int E, int R, int32_t *rank_idx) {
    int per = E / R;
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[t * K + k];
            int out;
            if (e == -1) {
                out = -1;
            } else if (e < -1 || e >= E) {
                out = -2;
            } else {
                int r = e / per;
                out = r;
                for (int j = 0; j < k; ++j) {
                    int ej = topk_idx[t * K + j];
                    if (ej >= 0 && ej < E && ej / per == r) {
                        out = -1; /* the rank was named earlier */
                        break;
                    }
                }
            }
            rank_idx[t * K + k] = out;
        }
    }
}

/* Local expand: row dst_row[t,k] of the per-expert layout receives the send
 * row of (t, rank of topk_idx[t,k]), i.e. send_dst[t*K+j] for the first j
 * naming that rank; the scale row goes along.  Entries with dst_row < 0 are
 * skipped. */
void orc_rank_expand(const int32_t *topk_idx, int T, int K, int E, int R,
                     const int32_t *send_dst, const int32_t *dst_row, int row_bytes,
                     int scale_bytes, const void *send_rows, const void *send_scales,
                     void *out_rows, void *out_scales) {
    int per = E / R;
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int d = dst_row[t * K + k];
            int e = topk_idx[t * K + k];
            if (d < 0 || e < 0 || e >= E) continue;
            int src = -1;
            for (int j = 0; j <= k && src < 0; ++j) {
                int ej = topk_idx[t * K + j];
                if (ej >= 0 && ej < E && ej / per == e / per) src = send_dst[t * K + j];
            }
            if (src < 0) continue;
            memcpy((uint8_t *)out_rows + (size_t)d * row_bytes,
                   (const uint8_t *)send_rows + (size_t)src * row_bytes, (size_t)row_bytes);
            if (scale_bytes)
                memcpy((uint8_t *)out_scales + (size_t)d * scale_bytes,
                       (const uint8_t *)send_scales + (size_t)src * scale_bytes, (size_t)scale_bytes);
        }
    }
}

/* ------------------------------------------------- MN-major scale layout */

/* Packed UE8M0 scale words re-laid "MN-major" for a grouped GEMM that loads
 * per-row scale factors with TMA: word p of every row is contiguous along the
 * rows, each column padded to a multiple of 4 rows (16 bytes).
 *   contiguous layout (rows = the row space's capacity):
 *       out[p * roundup(rows, 4) + r]                 = row_major[r * P + p]
 *   masked layout (row r = e * cap + s):
 *       out[(e * P + p) * roundup(cap, 4) + s]        = row_major[r * P + p]
 * Entries of the padding are not written. */
void orc_scales_mn_major(const int32_t *row_major, int rows, int P, int masked, int E,
                         int cap, int32_t *out) {
    if (masked) {
        int cap4 = (cap + 3) / 4 * 4;
        for (int e = 0; e < E; ++e)
            for (int s = 0; s < cap; ++s)
                for (int p = 0; p < P; ++p)
                    out[((size_t)e * P + p) * cap4 + s] = row_major[((size_t)e * cap + s) * P + p];
    } else {
        int rows4 = (rows + 3) / 4 * 4;
        for (int r = 0; r < rows; ++r)
            for (int p = 0; p < P; ++p) out[(size_t)p * rows4 + r] = row_major[(size_t)r * P + p];
    }
}

/* --------------------------------------------------------- masked repack */

/* slab[e, s, :] = rows[offset[e] + s, :] for s < min(count[e], cap), and the
 * same for the per-row scales; masked_m[e] = min(count[e], cap).  Slab rows at
 * or beyond masked_m[e] are not written.  count[e] > cap -> ORC_CAPACITY. */
int orc_masked_repack(const void *rows, const void *row_scales, int H, int quant,
                      const int32_t *offset, const int32_t *count, int E, int cap,
                      void *slab, void *slab_scales, int32_t *masked_m) {
    int status = ORC_OK;
    size_t row_bytes = quant == ORC_Q_NONE ? 2 * (size_t)H : (size_t)H;
    int G = H / 128;
    size_t scale_bytes = quant == ORC_Q_FP8_F32 ? 4 * (size_t)G
                         : quant == ORC_Q_FP8_UE8M0 ? 4 * (size_t)((G + 3) / 4)
                         : quant == ORC_Q_MXFP8 ? (size_t)(H / 32) : 0;
    for (int e = 0; e < E; ++e) {
        int n = count[e];
        if (n > cap) {
            n = cap;
            if (status < ORC_CAPACITY) status = ORC_CAPACITY;
        }
        masked_m[e] = n;
        for (int s = 0; s < n; ++s) {
            size_t src = (size_t)offset[e] + (size_t)s;
            size_t dst = (size_t)e * (size_t)cap + (size_t)s;
            memcpy((uint8_t *)slab + dst * row_bytes, (const uint8_t *)rows + src * row_bytes, row_bytes);
            if (scale_bytes)
                memcpy((uint8_t *)slab_scales + dst * scale_bytes,
                       (const uint8_t *)row_scales + src * scale_bytes, scale_bytes);
        }
    }
    return status;
}
