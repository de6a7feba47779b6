"""Per-rank deduplicated send layout, send-buffer dispatch and local expand on
the GPU, against the oracle; expand(send) must equal the direct dispatch."""
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

CASES = [
    workloads.CONFIGS["skewed_zipf"],  # R = 8 ranks of 16 experts, bf16
    workloads.Workload("dsv3_ranks", T=4096, H=7168, E=256, K=8, routing="grouped_sigmoid",
                       layout="contig", quant="fp8_ue8m0", align=128, R=8, seed=41),
    workloads.Workload("mx_ranks_ragged", T=777, H=640, E=96, K=6, routing="softmax",
                       layout="contig", quant="mxfp8", align=32, R=12, seed=42),
    workloads.Workload("f32_ranks_small", T=300, H=256, E=16, K=4, routing="softmax",
                       layout="contig", quant="fp8_f32", align=1, R=16, seed=43),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_rank_send_and_expand(w):
    case = gh.make_case(w)
    idx = case["idx"].copy()
    if w.name == "mx_ranks_ragged":  # unrouted entries and repeated experts too
        idx[::5, 1] = -1
        idx[::7, 2] = idx[::7, 0]
    idx_d = torch.from_numpy(idx).cuda()
    orc = oracle.default()
    RL, rank_idx = ep.ep_rank_layout(idx_d, w.E, w.R)
    L = ep.ep_layout(idx_d, w.E, kind="contig", align=w.align)
    send_rows, send_sc, _ = ep.ep_dispatch(RL, case["x_d"], w.quant)
    out_rows, out_sc = ep.ep_rank_expand(RL, L, idx_d, w.quant, send_rows, send_sc)
    direct_rows, direct_sc, _ = ep.ep_dispatch(L, case["x_d"], w.quant)
    torch.cuda.synchronize()

    assert np.array_equal(rank_idx.cpu().numpy(), orc.rank_ids(idx, w.E, w.R))
    ref = orc.rank_layout(idx, w.E, w.R, align=1)
    T, K = idx.shape
    assert int(RL.status.item()) == ref["status"] == 0
    assert np.array_equal(RL.expert_count.cpu().numpy(), ref["count"])
    assert np.array_equal(RL.expert_offset.cpu().numpy(), ref["offset"])
    assert np.array_equal(RL.dst_row.cpu().numpy()[:T * K].reshape(T, K), ref["dst_row"])
    assert np.array_equal(RL.row_src.cpu().numpy()[:ref["rows"]], ref["row_src"])
    # send buffer vs the oracle's dispatch into the send layout (valid rows)
    o_rows, o_sc, _ = orc.dispatch(case["x"], ref["dst_row"], ref["rows"], w.quant)
    n = ref["rows"]
    got = send_rows[:n].contiguous().view(torch.uint8).cpu().numpy()
    assert np.array_equal(got, o_rows.view(np.uint8).reshape(n, -1))
    if w.quant != "none":
        assert np.array_equal(send_sc[:n].cpu().numpy().view(np.uint32), o_sc.view(np.uint32))
    # expand == direct dispatch on every row the expert layout uses
    ref_e = orc.layout(idx, w.E, "contig", align=w.align)
    valid = torch.from_numpy(np.nonzero(ref_e["row_src"] >= 0)[0]).cuda()
    assert torch.equal(out_rows.index_select(0, valid).view(torch.uint8),
                       direct_rows.index_select(0, valid).view(torch.uint8))
    if w.quant != "none":
        assert torch.equal(out_sc.index_select(0, valid).view(torch.int32),
                           direct_sc.index_select(0, valid).view(torch.int32))
