"""ep_layout_dispatch: the layout and the dispatch in one call must give
bit-identical results to ep_layout followed by ep_dispatch, and match the
oracle, on both layout paths (the cluster kernel up to 16384 entries, the
histogram + assign kernels beyond)."""
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

W = workloads.Workload
CASES = [
    workloads.CONFIGS["qwen3_30b_a3b_decode"],
    workloads.CONFIGS["dsv3_decode"],
    workloads.CONFIGS["tiny"],
    W("fused_mx", T=300, H=2048, E=64, K=8, routing="softmax", layout="contig", quant="mxfp8",
      align=32, R=4, seed=81),
    W("fused_mn_masked", T=500, H=1024, E=40, K=6, routing="softmax", layout="masked",
      quant="fp8_ue8m0_mn", cap=90, seed=82),   # capacity overflow
    W("fused_f32_ragged", T=777, H=640, E=100, K=9, routing="softmax", layout="contig",
      quant="fp8_f32", align=16, seed=83),
    W("fused_bf16_big_h", T=40, H=16384, E=8, K=2, routing="softmax", layout="masked",
      quant="none", cap=40, seed=84),
    W("cluster_16000", T=2000, H=512, E=64, K=8, routing="softmax", layout="contig",
      quant="fp8_ue8m0", align=128, seed=85),   # 16000 entries: cluster layout of 4 rounds
    W("cluster_bad_over", T=900, H=512, E=64, K=8, routing="softmax", layout="masked",
      quant="fp8_ue8m0", cap=60, R=4, seed=86),  # bad ids and capacity overflow
    W("tiled_16800", T=2100, H=256, E=64, K=8, routing="softmax", layout="contig",
      quant="fp8_f32", align=128, seed=87),     # 16800 entries: histogram + assign kernels
]


def _alloc(w, L):
    rows = L.rows_capacity
    dev = torch.device("cuda")
    if w.quant == "none":
        rows_t = torch.full((max(rows, 1), w.H), gh.SENTINEL_BF16, dtype=torch.int16,
                            device=dev).view(torch.bfloat16)
    else:
        rows_t = torch.full((max(rows, 1), w.H), gh.SENTINEL_U8, dtype=torch.uint8, device=dev)
    sc = None if w.quant == "none" else ep.scale_buffer(L, w.H, w.quant)
    if sc is not None:
        sc.zero_()
    row_w = torch.zeros(max(rows, 1), dtype=torch.float32, device=dev)
    return rows_t, sc, row_w


def _arrays(L):
    used = int(L.expert_offset[-1].item())  # rows past offset[E] are never written
    return dict(dst_row=L.dst_row.cpu(), count=L.expert_count.cpu(), offset=L.expert_offset.cpu(),
                rank_rows=L.rank_rows.cpu(), status=L.status.cpu(),
                row_src=None if L.row_src is None else L.row_src[:used].cpu())


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_equals_two_calls_and_oracle(w):
    case = gh.make_case(w)
    idx = case["idx"].copy()
    if w.name in ("fused_f32_ragged", "cluster_bad_over"):  # unrouted entries and bad ids too
        idx[::7, 3] = -1
        idx[5, 0] = w.E + 2
        idx[w.T - 1, w.K - 1] = -9
    idx_d = torch.from_numpy(idx).cuda()
    case["idx"], case["idx_d"] = idx, idx_d
    # reference: the two calls
    L1 = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    r1, s1, rw1 = _alloc(w, L1)
    ep.ep_layout(idx_d, w.E, out=L1)
    ep.ep_dispatch(L1, case["x_d"], w.quant, out_rows=r1, out_scales=s1, topk_w=case["w_d"],
                   row_w=rw1)
    # one call
    L2 = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    r2, s2, rw2 = _alloc(w, L2)
    ep.ep_layout_dispatch(idx_d, L2, case["x_d"], w.quant, out_rows=r2, out_scales=s2,
                          topk_w=case["w_d"], row_w=rw2)
    torch.cuda.synchronize()
    a1, a2 = _arrays(L1), _arrays(L2)
    for k in a1:
        if a1[k] is not None:
            assert torch.equal(a1[k], a2[k]), f"layout array {k} differs"
    assert torch.equal(r1.view(torch.uint8), r2.view(torch.uint8)), "rows differ"
    if s1 is not None:
        assert torch.equal(s1.view(torch.int32), s2.view(torch.int32)), "scales differ"
    assert torch.equal(rw1.view(torch.int32), rw2.view(torch.int32)), "row weights differ"
    # and the oracle (layout, rows, scales, row weights)
    res = dict(L=L2, rows=L2.rows_capacity, out_rows=r2, out_scales=s2, row_w=rw2)
    ref = gh.check_layout(w, case, res)
    if w.quant != "fp8_ue8m0_mn":  # the MN-major word order has its own test file
        gh.check_dispatch(w, case, res, ref, sample_tokens=512)


def test_fused_graph_replay():
    """Captured once with combine in a CUDA graph, replayed on fresh inputs."""
    w = workloads.CONFIGS["qwen3_30b_a3b_decode"]
    dev = torch.device("cuda")
    idx_s = torch.zeros((w.T, w.K), dtype=torch.int32, device=dev)
    w_s = torch.zeros((w.T, w.K), dtype=torch.float32, device=dev)
    x_s = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device=dev)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, capacity=w.cap)
    rows = L.rows_capacity
    out_rows = torch.empty((rows, w.H), dtype=torch.uint8, device=dev)
    out_sc = ep.scale_buffer(L, w.H, w.quant)
    y = workloads.make_expert_outputs(rows, w.H, seed=5, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()

    def step():
        ep.ep_layout_dispatch(idx_s, L, x_s, w.quant, out_rows=out_rows, out_scales=out_sc,
                              stream=s)
        ep.ep_combine(L, y, w_s, out=out, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for seed in (31, 32):
        wi = w.with_(seed=seed)
        idx, wts, x = workloads.make_inputs(wi)
        idx_s.copy_(torch.from_numpy(idx))
        w_s.copy_(torch.from_numpy(wts))
        x_s.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        case = dict(idx=idx, w=wts, x=x)
        res = dict(L=L, rows=rows, out_rows=out_rows, out_scales=out_sc, row_w=None, y=y, out=out)
        ref = gh.check_layout(wi, case, res)
        gh.check_dispatch(wi, case, res, ref, check_row_w=False)
        assert gh.check_combine(wi, case, res, ref) == 1.0


QUANTS = ["none", "fp8_f32", "fp8_ue8m0", "mxfp8", "fp8_ue8m0_mn"]


@pytest.mark.parametrize("seed", range(24))
def test_fused_fuzz_equals_two_calls(seed):
    """Random decode-sized shapes (up to 8192 entries) with -1
    ids, repeated experts and small masked capacities: every output array
    equals ep_layout followed by ep_dispatch, and the one call's outputs equal
    the oracle's."""
    rng = np.random.default_rng(500 + seed)
    K = int(rng.integers(1, 33))
    T = int(rng.integers(1, 8192 // K + 1))
    E = int(rng.choice([1, 5, 16, 64, 128, 256, 361, 1024]))
    K = min(K, max(E, 1)) if E < K else K
    quant = QUANTS[seed % len(QUANTS)]
    H = int(rng.choice([128, 256, 1024, 2048, 7168, 32768] if quant != "none"
                       else [8, 264, 2048, 7168, 32768]))
    if H * T > 64 * 1024 * 1024:  # keep the buffers small
        T = max(1, 64 * 1024 * 1024 // H)
    layout = "masked" if rng.random() < 0.5 else "contig"
    cap = int(rng.integers(1, max(2, T * K // max(E, 1) * 2 + 2)))
    align = int(rng.choice([1, 4, 32, 128]))
    R = int(rng.choice([r for r in (1, 2, 4) if E % r == 0]))
    w = W(f"ffuzz{seed}", T=T, H=H, E=E, K=K, routing="softmax", layout=layout, quant=quant,
          align=align, cap=cap, R=R, seed=seed)
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    wts = rng.random((T, K)).astype(np.float32)
    x = workloads.make_x(w, rng)
    idx_d = torch.from_numpy(idx).cuda()
    w_d = torch.from_numpy(wts).cuda()
    x_d = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    outs = []
    for one_call in (False, True):
        L = ep.new_layout(T, K, E, layout, align=align, capacity=cap, num_ranks=R)
        r, s, rw = _alloc(w, L)
        if one_call:
            ep.ep_layout_dispatch(idx_d, L, x_d, quant, out_rows=r, out_scales=s, topk_w=w_d,
                                  row_w=rw)
        else:
            ep.ep_layout(idx_d, E, out=L)
            ep.ep_dispatch(L, x_d, quant, out_rows=r, out_scales=s, topk_w=w_d, row_w=rw)
        torch.cuda.synchronize()
        outs.append((_arrays(L), r, s, rw))
    (a1, r1, s1, rw1), (a2, r2, s2, rw2) = outs
    for k in a1:
        if a1[k] is not None:
            assert torch.equal(a1[k], a2[k]), f"layout array {k} differs"
    assert torch.equal(r1.view(torch.uint8), r2.view(torch.uint8)), "rows differ"
    if s1 is not None:
        assert torch.equal(s1.view(torch.int32), s2.view(torch.int32)), "scales differ"
    assert torch.equal(rw1.view(torch.int32), rw2.view(torch.int32)), "row weights differ"
    # the one call against the oracle too: every layout array and status, every
    # valid row, scale word and row weight, sentinels on the rows left empty
    case = dict(idx=idx, w=wts, x=x)
    res = dict(L=L, rows=L.rows_capacity, out_rows=r2, out_scales=s2, row_w=rw2)
    ref = gh.check_layout(w, case, res)
    if quant == "fp8_ue8m0_mn":
        gh.check_dispatch_mn(w, case, L, r2, s2, ref)
    else:
        gh.check_dispatch(w, case, res, ref)


@pytest.mark.parametrize("layout", ["contig", "masked"])
def test_fused_zero_tokens(layout):
    """No tokens: the layout arrays say so (zero counts, zero rank rows,
    offsets of empty experts, status OK) and nothing else is written."""
    E, K, H = 16, 4, 256
    dev = torch.device("cuda")
    L = ep.new_layout(0, K, E, layout, align=128, capacity=8, num_ranks=4)
    w = W("zero", T=0, H=H, E=E, K=K, routing="softmax", layout=layout, quant="fp8_f32",
          align=128, cap=8, R=4, seed=0)
    r, s, rw = _alloc(w, L)
    r_before = r.clone()
    L.expert_count.fill_(7)
    L.rank_rows.fill_(7)
    L.status.fill_(5)
    idx_d = torch.empty((0, K), dtype=torch.int32, device=dev)
    x_d = torch.empty((0, H), dtype=torch.bfloat16, device=dev)
    ep.ep_layout_dispatch(idx_d, L, x_d, "fp8_f32", out_rows=r, out_scales=s)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    assert not L.expert_count.any() and not L.rank_rows.any()
    want = [e * 8 for e in range(E + 1)] if layout == "masked" else [0] * (E + 1)
    assert L.expert_offset.cpu().tolist() == want
    assert torch.equal(r, r_before)
