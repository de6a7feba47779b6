"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Every mutant is a one-line edit of ``oracle/oracle.c`` compiled into a temporary
library; the real oracle is untouched.  A mutant that no pin rejects would mean
the pins leave that part of the oracle unchecked.
"""
import os
import shutil

import numpy as np
import pytest

import oracle
from tests import pins

MUTANTS = {
    "bf16_ties_away": ("(rem == 0x8000u && ((lo >> 16) & 1u))", "(rem == 0x8000u)"),
    "e4m3_truncate": ("nearbyint((2.0 * f - 1.0) * 8.0)", "floor((2.0 * f - 1.0) * 8.0)"),
    "e4m3_subnormal_step": ("nearbyint(a * 512.0)", "nearbyint(a * 256.0)"),
    "e4m3_bias": ("((e + 7) << 3)", "((e + 8) << 3)"),
    "e4m3_no_satfinite": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
                          "if (a >= 480.0) return (uint8_t)(sign | 0x7F);"),
    "scale_wrong_max": ("fmaxf(group_amax(x, n), 1e-4f) / 448.0f;\n    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) / s);",
                        "fmaxf(group_amax(x, n), 1e-4f) / 240.0f;\n    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) / s);"),
    "amax_signed": ("float v = fabsf(orc_bf16_to_float(x[i]));", "float v = orc_bf16_to_float(x[i]);"),
    "ue8m0_floor": ("+ ((bits & 0x007FFFFFu) != 0u)", "+ 0"),
    "mx_ceil_scale": ("e = ex - 1 + 127;", "e = ex + 127;"),
    "mx_emax7": ("int byte = e - 8 > 0 ? e - 8 : 0;", "int byte = e - 7 > 0 ? e - 7 : 0;"),
    "mx_scale_byte_layout": ("memcpy((uint8_t *)out_scales + (size_t)dst * (H / 32), mx, (size_t)(H / 32));",
                             "memcpy((uint8_t *)out_scales + (size_t)dst * (H / 32), mx + (H > 32), (size_t)(H / 32 - (H > 32)));"),
    "mn_major_unaligned": ("int rows4 = (rows + 3) / 4 * 4;", "int rows4 = rows;"),
    "mn_major_swapped": ("out[((size_t)e * P + p) * cap4 + s]", "out[((size_t)p * E + e) * cap4 + s]"),
    "rank_no_dedup": ("                        out = -1; /* the rank was named earlier */", "                        out = r;"),
    "rank_expand_wrong_source": ("for (int j = 0; j <= k && src < 0; ++j)", "for (int j = k; j <= k && src < 0; ++j)"),
    "route_ties_high": ("return va > vb || (va == vb && a < b);", "return va > vb || (va == vb && a > b);"),
    "route_group_top1": ("gscore[g] = (double)((float)score[g * gs + two[0]] + (float)score[g * gs + two[1]]);",
                         "gscore[g] = (double)((float)score[g * gs + two[0]]);"),
    "route_no_renorm": ("topk_w[t * K + j] = sig[pick[j]] / sum;", "topk_w[t * K + j] = sig[pick[j]];"),
    "route_no_bias": ("c32[e] = s32 + (bias ? bias[e] : 0.0f);", "c32[e] = s32;"),
    "layout_no_padding": ("offset[e] + round_up(count[e], align)", "offset[e] + count[e]"),
    "layout_k_descending": ("for (int k = 0; k < K; ++k) {\n            int i = t * K + k;",
                            "for (int k = K - 1; k >= 0; --k) {\n            int i = t * K + k;"),
    "layout_no_capacity_status": ("if (masked && slot >= cap) {\n                if (status < ORC_CAPACITY) status = ORC_CAPACITY;",
                                  "if (masked && slot >= cap) {\n                ;"),
    "dispatch_scale_shift": ("memcpy((float *)out_scales + (size_t)dst * G, sc, sizeof(float) * (size_t)G);",
                             "memcpy((float *)out_scales + (size_t)dst * G, sc + (G > 1), sizeof(float) * (size_t)(G - (G > 1)));"),
    "ue8m0_pad_byte": ("eb[b] = 127;", "eb[b] = 0;"),
    "combine_dropped_term": ("acc = acc + p;", "acc = p;"),
    "combine_double_reduce": ("acc = acc + p;", "acc = acc + p + p;"),
    "layout_bad_id_silent": ("if (status < ORC_BAD_EXPERT_ID) status = ORC_BAD_EXPERT_ID;", ";"),
    "layout_rank_rows_shifted": ("for (int e = r * per; e < (r + 1) * per; ++e) s += count[e];",
                                 "for (int e = r * per + 1; e <= (r + 1) * per && e < E; ++e) s += count[e];"),
    "repack_slots_reversed": ("size_t src = (size_t)offset[e] + (size_t)s;",
                              "size_t src = (size_t)offset[e] + (size_t)(n - 1 - s);"),
    "combine_fused_multiply_add": ("acc = acc + p;",
                                   "acc = fmaf(topk_w[t * K + k], orc_bf16_to_float(y[(size_t)dst * H + h]), acc);"),
    "combine_transposed_w": ("float p = topk_w[t * K + k]", "float p = topk_w[k * T + t < T * K ? k * T + t : 0]"),
    "repack_masked_m_unclamped": ("masked_m[e] = n;", "masked_m[e] = count[e];"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur once"
    d = tmp_path / name
    d.mkdir()
    shutil.copy(oracle.HDR, d / "oracle.h")
    (d / "oracle.c").write_text(src.replace(old, new))
    return oracle.Oracle(oracle.compile_oracle(str(d / "oracle.c"), str(d / "liboracle.so"),
                                               include_dir=str(d)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    orc = _build_mutant(tmp_path, name)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc, np.random.default_rng(1234))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin rejects the mutant {name}"
