"""The decode sequence captured once in a CUDA graph and replayed on new inputs.

Fixed-capacity shapes make decode graph-capturable (SGLang PR "[Feature] Add
DeepEPv2 (ElasticBuffer) MoE A2A backend", section "Motivation"); the library
never synchronises or allocates, so layout -> dispatch -> combine (and the
masked repack) can be captured as they are.  Every replay must match the oracle
on that replay's inputs.
"""
import numpy as np
import pytest
import torch

import workloads
from combine_expert_histogram_gb300 import binding as ep
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.mark.parametrize("name", ["dsv3_decode", "qwen3_30b_a3b_decode", "skewed_zipf"])
def test_graph_replay_matches_oracle(name):
    w = workloads.CONFIGS[name]
    dev = torch.device("cuda")
    idx_s = torch.zeros((w.T, w.K), dtype=torch.int32, device=dev)
    w_s = torch.zeros((w.T, w.K), dtype=torch.float32, device=dev)
    x_s = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device=dev)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    rows = L.rows_capacity
    quant = w.quant
    out_rows = torch.empty((rows, w.H), device=dev,
                           dtype=torch.bfloat16 if quant == "none" else torch.uint8)
    out_scales = None
    if quant != "none":
        out_scales = torch.empty((rows, ep.ep_scale_cols(w.H, quant)), device=dev,
                                 dtype=torch.float32 if quant == "fp8_f32" else torch.int32)
    y = workloads.make_expert_outputs(rows, w.H, seed=5, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)

    s = torch.cuda.Stream()
    # warm-up outside capture (first launches may load modules)
    with torch.cuda.stream(s):
        ep.ep_layout(idx_s, w.E, out=L, stream=s)
        ep.ep_dispatch(L, x_s, quant, out_rows=out_rows, out_scales=out_scales, stream=s)
        ep.ep_combine(L, y, w_s, out=out, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ep.ep_layout(idx_s, w.E, out=L, stream=s)
        ep.ep_dispatch(L, x_s, quant, out_rows=out_rows, out_scales=out_scales, stream=s)
        ep.ep_combine(L, y, w_s, out=out, stream=s)

    for seed in (21, 22):
        wi = w.with_(seed=seed)
        idx, wts, x = workloads.make_inputs(wi)
        idx_s.copy_(torch.from_numpy(idx))
        w_s.copy_(torch.from_numpy(wts))
        x_s.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        case = dict(idx=idx, w=wts, x=x)
        res = dict(L=L, rows=rows, out_rows=out_rows, out_scales=out_scales,
                   row_w=None, y=y, out=out)
        ref = gh.check_layout(wi, case, res)
        gh.check_dispatch(wi, case, res, ref, sample_tokens=512, check_row_w=False)
        assert gh.check_combine(wi, case, res, ref, sample_tokens=512) == 1.0


FIRST_CALL_IN_CAPTURE = """
import sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import oracle
import workloads
from combine_expert_histogram_gb300 import binding as ep
from tests import gpu_harness as gh
for name in ("qwen3_30b_a3b_decode", "dsv3_prefill"):
    w = workloads.CONFIGS[name]
    if name == "dsv3_prefill":
        w = w.with_(T=4096, name="dsv3_prefill_T4096")   # the tiled layout path
    case = gh.make_case(w)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R)
    rows = torch.empty((L.rows_capacity, w.H), dtype=torch.uint8, device="cuda")
    sc = ep.scale_buffer(L, w.H, w.quant)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):  # the library's first launches of these kernels
        ep.ep_layout(case["idx_d"], w.E, out=L, stream=s)
        ep.ep_dispatch(L, case["x_d"], w.quant, out_rows=rows, out_scales=sc, stream=s)
    g.replay()
    torch.cuda.synchronize()
    res = dict(L=L, rows=L.rows_capacity, out_rows=rows, out_scales=sc, row_w=None)
    ref = gh.check_layout(w, case, res)
    gh.check_dispatch(w, case, res, ref, check_row_w=False)
    print("ok", name)
"""


def test_first_library_call_inside_graph_capture():
    """In a fresh process, the layout and dispatch kernels are first launched
    while a CUDA graph is being captured (the per-device queries and kernel
    attributes of the first launch happen inside the capture); the replayed
    graph matches the oracle, on the cluster and on the tiled layout path."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", FIRST_CALL_IN_CAPTURE.format(root=root)], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 2
