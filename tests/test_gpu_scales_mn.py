"""UE8M0 scale words written MN-major (TMA-aligned columns) by dispatch and
by the masked repack, against the oracle's re-layout of its row-major words."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_expert_histogram_gb300 import binding as ep
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SENT = 0x5A5A5A5A


def _mn_index(r, p, P, layout, stride, cap):
    if layout == "masked":
        return ((r // cap) * P + p) * stride + (r % cap)
    return p * stride + r


@pytest.mark.parametrize("layout,H", [("contig", 7168), ("masked", 7168), ("contig", 640),
                                      ("masked", 384)])
def test_dispatch_writes_mn_major_scales(layout, H):
    w = workloads.Workload("mn", T=1500, H=H, E=64, K=8, routing="softmax", layout=layout,
                           quant="fp8_ue8m0_mn", align=128, cap=1500, seed=31)
    case = gh.make_case(w)
    L = ep.ep_layout(case["idx_d"], w.E, kind=layout, align=w.align, capacity=w.cap)
    sc = ep.scale_buffer(L, H, "fp8_ue8m0_mn")
    sc.fill_(SENT)
    rows_t, _, _ = ep.ep_dispatch(L, case["x_d"], "fp8_ue8m0_mn", out_scales=sc)
    torch.cuda.synchronize()
    assert sc.numel() == ep.ep_scale_words(L, H, "fp8_ue8m0_mn")
    orc = oracle.default()
    ref = orc.layout(case["idx"], w.E, layout, align=w.align, cap=w.cap)
    cap_rows = L.rows_capacity
    o_rows, o_sc, _ = orc.dispatch(case["x"], ref["dst_row"], cap_rows, "fp8_ue8m0")
    mn = orc.scales_mn_major(o_sc, layout, E=w.E, cap=w.cap, fill=SENT)
    got = sc.reshape(-1).cpu().numpy()
    assert got.size == mn.size
    P = o_sc.shape[1]
    stride = (w.cap + 3) // 4 * 4 if layout == "masked" else (cap_rows + 3) // 4 * 4
    valid = np.nonzero(ref["row_src"] >= 0)[0]
    idx = np.array([_mn_index(r, p, P, layout, stride, w.cap) for r in valid for p in range(P)])
    assert np.array_equal(got[idx], mn[idx]), "MN-major scale words differ"
    untouched = np.ones(got.size, dtype=bool)
    untouched[idx] = False
    assert (got[untouched] == SENT).all()
    # the rows themselves are the plain UE8M0 rows
    assert np.array_equal(rows_t[:ref["rows"]].cpu().numpy()[valid], o_rows[valid])


def test_masked_repack_mn_major():
    w = workloads.CONFIGS["dsv3_decode"]
    case = gh.make_case(w)
    q = "fp8_ue8m0_mn"
    Lc = ep.ep_layout(case["idx_d"], w.E, kind="contig", align=128)
    rows_c, sc_c, _ = ep.ep_dispatch(Lc, case["x_d"], q)
    slab, slab_sc, mm = ep.ep_masked_repack(Lc, rows_c, sc_c, q, w.cap)
    Lm = ep.ep_layout(case["idx_d"], w.E, kind="masked", capacity=w.cap)
    rows_m, sc_m, _ = ep.ep_dispatch(Lm, case["x_d"], q)
    torch.cuda.synchronize()
    assert tuple(slab_sc.shape) == tuple(sc_m.shape)
    P = sc_m.shape[1]
    m = mm.cpu().numpy()
    valid_slot = torch.from_numpy(np.arange(sc_m.shape[2])[None, :] < m[:, None]).cuda()
    a = slab_sc.masked_select(valid_slot[:, None, :].expand_as(slab_sc))
    b = sc_m.masked_select(valid_slot[:, None, :].expand_as(sc_m))
    assert torch.equal(a, b)
    assert P == (w.H // 128 + 3) // 4
