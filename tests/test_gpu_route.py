"""ep_route_topk on the GPU against the oracle router.

Indices: softmax selection ranks the logits, so it must match exactly (exact
ties included).  The grouped sigmoid selection ranks fp32 sigmoid scores; the
GPU's expf and the host's expf may differ in the last place, so a token may
differ only where the decision is a near-tie at fp32 resolution (checked in
fp64), and such tokens must stay rare.  Weights: within 2^-16 relative of the
oracle's fp64 weights (a handful of fp32 roundings of values in (0, 1]).
"""
import numpy as np
import pytest
import torch

import oracle

from combine_expert_histogram_gb300 import binding as ep

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

W_TOL = 2.0 ** -16


@pytest.mark.parametrize("T,E,K,ties", [(256, 128, 8, False), (16384, 256, 8, False),
                                        (512, 64, 6, True), (300, 1024, 32, False),
                                        (100, 4, 4, True), (200, 32, 3, True),
                                        (150, 40, 7, True), (100, 1000, 8, False)])
def test_softmax_route(T, E, K, ties):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        lg = np.round(lg * 2) / 2
    idx, w = ep.ep_route_topk(torch.from_numpy(lg).cuda(), K, "softmax")
    torch.cuda.synchronize()
    o_idx, o_w, _ = oracle.default().route_topk(lg, K, "softmax")
    assert np.array_equal(idx.cpu().numpy(), o_idx)
    g = w.cpu().numpy().astype(np.float64)
    assert (np.abs(g - o_w) <= W_TOL * np.abs(o_w)).all()


def _margins(lg, bias, G, TG, K):
    """fp64 gaps at the group and the expert decision boundaries, per token."""
    s = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
    c = s + bias.astype(np.float64)
    T, E = c.shape
    gs = E // G
    top2 = -np.sort(-c.reshape(T, G, gs), axis=2)[:, :, :2].sum(axis=2)
    gsorted = -np.sort(-top2, axis=1)
    g_gap = gsorted[:, TG - 1] - gsorted[:, TG] if TG < G else np.full(T, np.inf)
    keep = np.argsort(-top2, axis=1, kind="stable")[:, :TG]
    mask = np.zeros((T, G), dtype=bool)
    np.put_along_axis(mask, keep, True, axis=1)
    cm = np.where(np.repeat(mask, gs, axis=1), c, -np.inf)
    csorted = -np.sort(-cm, axis=1)
    e_gap = csorted[:, K - 1] - csorted[:, K] if K < TG * gs else np.full(T, np.inf)
    return np.minimum(g_gap, e_gap)


@pytest.mark.parametrize("T,E,K,G,TG", [(1024, 256, 8, 8, 4), (16384, 256, 8, 8, 4),
                                        (500, 64, 6, 4, 2), (200, 1024, 32, 32, 8),
                                        (300, 32, 4, 16, 4), (400, 128, 8, 1, 1),
                                        # shapes outside the register path (shared memory)
                                        (300, 96, 6, 4, 2), (250, 48, 5, 3, 2)])
def test_grouped_sigmoid_route(T, E, K, G, TG):
    rng = np.random.default_rng(T * 7 + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    idx, w = ep.ep_route_topk(torch.from_numpy(lg).cuda(), K, "grouped_sigmoid",
                              bias=torch.from_numpy(bias).cuda(), n_group=G, topk_group=TG)
    torch.cuda.synchronize()
    o_idx, o_w, _ = oracle.default().route_topk(lg, K, "grouped_sigmoid", bias=bias,
                                                n_group=G, topk_group=TG)
    gi = idx.cpu().numpy()
    diff = np.nonzero((gi != o_idx).any(axis=1))[0]
    if diff.size:
        m = _margins(lg, bias, G, TG, K)
        assert (m[diff] < 1e-5).all(), "selection differs away from an fp32 near-tie"
        assert diff.size <= max(2, T // 1000)
    same = np.setdiff1d(np.arange(T), diff)
    g = w.cpu().numpy().astype(np.float64)[same]
    assert (np.abs(g - o_w[same]) <= W_TOL * np.abs(o_w[same])).all()
    # picks are distinct on every row and in range
    assert (gi >= 0).all() and (gi < E).all()
    srt = np.sort(gi, axis=1)
    assert (srt[:, 1:] != srt[:, :-1]).all(), "a token picked one expert twice"
    # every pick lies in a kept group: the picks span at most topk_group
    # groups, and those groups are the top-scoring ones (fp64 group scores)
    # on every row whose group decision is not an fp32 near-tie
    gsz = E // G
    pick_groups = gi // gsz
    n_groups = np.array([len(set(r)) for r in pick_groups])
    assert (n_groups <= TG).all(), "picks span more groups than topk_group"
    s64 = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
    c64 = s64 + bias.astype(np.float64)
    top2 = -np.sort(-c64.reshape(T, G, gsz), axis=2)[:, :, :2].sum(axis=2)
    gsorted = -np.sort(-top2, axis=1)
    g_gap = gsorted[:, TG - 1] - gsorted[:, TG] if TG < G else np.full(T, np.inf)
    kept = np.zeros((T, G), dtype=bool)
    np.put_along_axis(kept, np.argsort(-top2, axis=1, kind="stable")[:, :TG], True, axis=1)
    in_kept = np.take_along_axis(kept, pick_groups, axis=1).all(axis=1)
    clear = g_gap >= 1e-5
    assert in_kept[clear].all(), "a pick lies outside the kept groups"


# 2048 tokens: a router grid of 512 CTAs, launched plainly; 256 tokens: 64
# CTAs, launched as a programmatic dependent that lets the layout launch
# early (the layout reads topk_idx only after its own wait)
@pytest.mark.parametrize("T,E,mode,layout", [(2048, 256, "grouped_sigmoid", "contig"),
                                             (256, 128, "softmax", "masked")])
def test_route_then_layout_chain(T, E, mode, layout):
    """Router output straight into layout, dispatch and combine (oracle on the same ids)."""
    from tests import gpu_harness as gh
    import workloads
    K, H = 8, 1024
    rng = np.random.default_rng(3)
    lg = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    bias = torch.from_numpy((rng.standard_normal(E) * 0.1).astype(np.float32)).cuda()
    w = workloads.Workload("chain", T=T, H=H, E=E, K=K, routing=mode, layout=layout,
                           quant="fp8_f32", align=128, cap=T)
    x = workloads.make_x(w)
    x_d = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    # every input is on the device before the router runs, and nothing waits
    # on the host between the router and the layout
    if mode == "softmax":
        idx_d, w_d = ep.ep_route_topk(lg, K, "softmax")
    else:
        idx_d, w_d = ep.ep_route_topk(lg, K, "grouped_sigmoid", bias=bias, n_group=8,
                                      topk_group=4)
    case = dict(x=x, idx_d=idx_d, w_d=w_d, x_d=x_d)
    g = gh.run_gpu(w, case)
    case["idx"], case["w"] = idx_d.cpu().numpy(), w_d.cpu().numpy()
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0
