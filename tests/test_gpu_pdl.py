"""Programmatic dependent launch: a kernel that starts while its predecessor
still runs must read that predecessor's results only after waiting for it.

The layout, dispatch, combine and rank kernels are launched as programmatic
dependents (the layout's first kernel waits for its predecessor before
anything else), and dispatch and combine let their dependents launch at their
start.  Here the stream is first held behind a long fill, so that the
library's launches queue back to back and every programmatic edge is live
(dispatch starts while the layout runs, combine while dispatch runs, the next
step's layout while combine runs).
The layout arrays and the outputs still hold an earlier call's results for
other inputs -- valid-looking rows, not garbage -- so a read issued before its
wait lands a row in the wrong place and the oracle check fails.
"""
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
    workloads.CONFIGS["dsv3_decode"],            # masked, UE8M0, fill CTAs, two layout kernels
    workloads.CONFIGS["qwen3_30b_a3b_decode"],   # masked, fp32 scales
    W("one_kernel_layout", T=96, H=512, E=64, K=8, routing="softmax", layout="contig",
      quant="fp8_f32", align=32, seed=61),       # T*K <= 1024: single layout kernel
    W("prefill_4k", T=4096, H=7168, E=256, K=8, routing="grouped_sigmoid", layout="contig",
      quant="fp8_f32", align=128, seed=62),      # TMA-stored fp32 scale rows
    W("mx_contig", T=1500, H=2048, E=128, K=8, routing="softmax", layout="contig",
      quant="mxfp8", align=128, seed=63),
    W("bf16_zipf", T=2048, H=4096, E=128, K=8, routing="zipf", layout="contig",
      quant="none", align=128, R=8, seed=64),
]


class Held:
    """Keeps `stream` busy for about a millisecond so later launches queue."""

    def __init__(self, stream):
        self.stream = stream
        self.big = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def hold(self):
        with torch.cuda.stream(self.stream):
            for i in range(12):
                self.big.fill_(i)


def _load(case, idx_d, w_d, x_d, w):
    idx, wts, x = workloads.make_inputs(w)
    idx_d.copy_(torch.from_numpy(idx))
    w_d.copy_(torch.from_numpy(wts))
    x_d.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
    case.update(idx=idx, w=wts, x=x)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layout_dispatch_combine_queued(w):
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    held = Held(s)
    idx_d = torch.empty((w.T, w.K), dtype=torch.int32, device=dev)
    w_d = torch.empty((w.T, w.K), dtype=torch.float32, device=dev)
    x_d = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    rows = L.rows_capacity
    out_rows = torch.empty((rows, w.H), device=dev,
                           dtype=torch.bfloat16 if w.quant == "none" else torch.uint8)
    out_scales = None if w.quant == "none" else ep.scale_buffer(L, w.H, w.quant)
    row_w = torch.empty(rows, dtype=torch.float32, device=dev)
    y = workloads.make_expert_outputs(rows, w.H, seed=5, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    case = {}

    def chain():
        ep.ep_layout(idx_d, w.E, out=L, stream=s)
        ep.ep_dispatch(L, x_d, w.quant, out_rows=out_rows, out_scales=out_scales,
                       topk_w=w_d, row_w=row_w, stream=s)
        ep.ep_combine(L, y, w_d, out=out, stream=s)

    for seed in (w.seed + 100, w.seed):  # the first call leaves stale, valid-looking results
        _load(case, idx_d, w_d, x_d, w.with_(seed=seed))
        torch.cuda.synchronize()
        held.hold()
        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
    res = dict(L=L, rows=rows, out_rows=out_rows, out_scales=out_scales, row_w=row_w, y=y,
               out=out)
    ref = gh.check_layout(w, case, res)
    gh.check_dispatch(w, case, res, ref, check_row_w=True, check_empty=False)
    assert gh.check_combine(w, case, res, ref) == 1.0


@pytest.mark.parametrize("w", [CASES[0], CASES[3]], ids=lambda w: w.name)
def test_layout_then_combine_queued(w):
    """Combine directly after the layout: its wait is on the layout's last kernel."""
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    held = Held(s)
    idx_d = torch.empty((w.T, w.K), dtype=torch.int32, device=dev)
    w_d = torch.empty((w.T, w.K), dtype=torch.float32, device=dev)
    x_d = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    y = workloads.make_expert_outputs(L.rows_capacity, w.H, seed=9, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    case = {}
    for seed in (w.seed + 200, w.seed + 1):
        _load(case, idx_d, w_d, x_d, w.with_(seed=seed))
        torch.cuda.synchronize()
        held.hold()
        with torch.cuda.stream(s):
            ep.ep_layout(idx_d, w.E, out=L, stream=s)
            ep.ep_combine(L, y, w_d, out=out, stream=s)
        torch.cuda.synchronize()
    res = dict(L=L, rows=L.rows_capacity, y=y, out=out)
    ref = gh.check_layout(w, case, res)
    assert gh.check_combine(w, case, res, ref) == 1.0


def test_rank_send_expand_queued():
    """rank layout -> dispatch into the send layout -> expand, all queued."""
    w = W("dsv3_ranks_q", T=2048, H=7168, E=256, K=8, routing="grouped_sigmoid",
          layout="contig", quant="fp8_ue8m0", align=128, R=8, seed=65)
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    held = Held(s)
    idx_d = torch.empty((w.T, w.K), dtype=torch.int32, device=dev)
    w_d = torch.empty((w.T, w.K), dtype=torch.float32, device=dev)
    x_d = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    RL = ep.new_layout(w.T, w.K, w.R, "contig", align=1)
    rank_idx = torch.empty((w.T, w.K), dtype=torch.int32, device=dev)
    L = ep.new_layout(w.T, w.K, w.E, "contig", align=w.align)
    send_rows = torch.empty((RL.rows_capacity, w.H), dtype=torch.uint8, device=dev)
    send_sc = ep.scale_buffer(RL, w.H, w.quant)
    out_rows = torch.empty((L.rows_capacity, w.H), dtype=torch.uint8, device=dev)
    out_sc = ep.scale_buffer(L, w.H, w.quant)
    case = {}
    for seed in (w.seed + 300, w.seed):
        _load(case, idx_d, w_d, x_d, w.with_(seed=seed))
        torch.cuda.synchronize()
        held.hold()
        with torch.cuda.stream(s):
            ep.ep_layout(idx_d, w.E, kind="contig", align=w.align, out=L, stream=s)
            ep.ep_rank_layout(idx_d, w.E, w.R, out=RL, rank_idx=rank_idx, stream=s)
            ep.ep_dispatch(RL, x_d, w.quant, out_rows=send_rows, out_scales=send_sc, stream=s)
            ep.ep_rank_expand(RL, L, idx_d, w.quant, send_rows, send_sc, out_rows=out_rows,
                              out_scales=out_sc, stream=s)
        torch.cuda.synchronize()
    orc = oracle.default()
    ref = orc.layout(case["idx"], w.E, "contig", align=w.align)
    o_rows, o_sc, _ = orc.dispatch(case["x"], ref["dst_row"], ref["rows"], w.quant)
    valid = np.nonzero(ref["row_src"] >= 0)[0]
    sel = torch.from_numpy(valid).to(dev)
    assert np.array_equal(out_rows.index_select(0, sel).cpu().numpy(), o_rows[valid])
    assert np.array_equal(out_sc.index_select(0, sel).cpu().numpy().view(np.uint32),
                          o_sc[valid].view(np.uint32))


@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[2], CASES[3]], ids=lambda w: w.name)
def test_back_to_back_steps_share_layout_arrays(w):
    """Two whole steps queued back to back on the same layout arrays: step A's
    combine still reads dst_row while step B's layout is next in line to
    rewrite it, and every kernel triggers its dependents early.  Each step must
    match the oracle on its own inputs."""
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    held = Held(s)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    rows = L.rows_capacity
    y = workloads.make_expert_outputs(rows, w.H, seed=11, device=dev)
    steps = []
    for seed in (w.seed + 400, w.seed + 401):
        idx, wts, x = workloads.make_inputs(w.with_(seed=seed))
        steps.append(dict(
            case=dict(idx=idx, w=wts, x=x),
            idx_d=torch.from_numpy(idx).to(dev), w_d=torch.from_numpy(wts).to(dev),
            x_d=torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16),
            out_rows=torch.empty((rows, w.H), device=dev,
                                 dtype=torch.bfloat16 if w.quant == "none" else torch.uint8),
            out_scales=None if w.quant == "none" else ep.scale_buffer(L, w.H, w.quant),
            out=torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)))
    torch.cuda.synchronize()
    held.hold()
    with torch.cuda.stream(s):
        for st in steps:
            ep.ep_layout(st["idx_d"], w.E, out=L, stream=s)
            ep.ep_dispatch(L, st["x_d"], w.quant, out_rows=st["out_rows"],
                           out_scales=st["out_scales"], stream=s)
            ep.ep_combine(L, y, st["w_d"], out=st["out"], stream=s)
    torch.cuda.synchronize()
    orc = oracle.default()
    for st in steps:
        ref = orc.layout(st["case"]["idx"], w.E, w.layout, align=w.align, cap=w.cap, R=w.R)
        res = dict(out_rows=st["out_rows"], out_scales=st["out_scales"], row_w=None, y=y,
                   out=st["out"])
        gh.check_dispatch(w, st["case"], res, ref, check_row_w=False, check_empty=False)
        assert gh.check_combine(w, st["case"], res, ref) == 1.0
    # the arrays hold the second step's layout
    assert gh.check_layout(w, steps[1]["case"], dict(L=L, rows=rows)) is not None


def test_three_stream_pipeline_matches_synchronous():
    """The end-to-end pattern: uploads on one stream, the three calls on a
    second behind event waits, downloads on a third, two input sets in flight
    alternately.  A programmatic launch on the compute stream must still wait
    for the upload it depends on; every step must give the bytes a plain
    synchronous run of the same inputs gives."""
    w = CASES[3].with_(T=2048)
    dev = torch.device("cuda")
    hosts = []
    for seed in (w.seed + 500, w.seed + 501):
        idx, wts, x = workloads.make_inputs(w.with_(seed=seed))
        hosts.append(dict(idx=torch.from_numpy(idx).pin_memory(),
                          w=torch.from_numpy(wts).pin_memory(),
                          x=torch.from_numpy(x.view(np.int16)).pin_memory()))
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align)
    rows = L.rows_capacity
    y = workloads.make_expert_outputs(rows, w.H, seed=13, device=dev)
    out_rows = torch.empty((rows, w.H), dtype=torch.uint8, device=dev)
    sc = ep.scale_buffer(L, w.H, w.quant)
    ref = []
    for h in hosts:
        ep.ep_layout(h["idx"].to(dev), w.E, out=L)
        ep.ep_dispatch(L, h["x"].to(dev).view(torch.bfloat16), w.quant, out_rows=out_rows,
                       out_scales=sc)
        ref.append(ep.ep_combine(L, y, h["w"].to(dev)).view(torch.int16).cpu())
    torch.cuda.synchronize()
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    bufs = [dict(idx=torch.empty((w.T, w.K), dtype=torch.int32, device=dev),
                 w=torch.empty((w.T, w.K), dtype=torch.float32, device=dev),
                 x=torch.empty((w.T, w.H), dtype=torch.int16, device=dev),
                 out=torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev))
            for _ in range(2)]
    n = 8
    got = [torch.empty((w.T, w.H), dtype=torch.int16).pin_memory() for _ in range(n)]
    done, fetched = {}, {}
    for i in range(n):
        b, h = bufs[i % 2], hosts[i % 2]
        if i >= 2:
            up.wait_event(done[i - 2])       # the buffer's previous step has read it
        with torch.cuda.stream(up):
            for k in ("idx", "w", "x"):
                b[k].copy_(h[k], non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up)
        comp.wait_event(loaded)
        if i >= 2:
            comp.wait_event(fetched[i - 2])  # its previous output has been read back
        with torch.cuda.stream(comp):
            ep.ep_layout(b["idx"], w.E, out=L, stream=comp)
            ep.ep_dispatch(L, b["x"].view(torch.bfloat16), w.quant, out_rows=out_rows,
                           out_scales=sc, stream=comp)
            ep.ep_combine(L, y, b["w"], out=b["out"], stream=comp)
            done[i] = torch.cuda.Event()
            done[i].record(comp)
        down.wait_event(done[i])
        with torch.cuda.stream(down):
            got[i].copy_(b["out"].view(torch.int16), non_blocking=True)
            fetched[i] = torch.cuda.Event()
            fetched[i].record(down)
    torch.cuda.synchronize()
    bad = [i for i in range(n) if not torch.equal(got[i], ref[i % 2])]
    assert not bad, f"pipelined steps {bad} differ from the synchronous run"
