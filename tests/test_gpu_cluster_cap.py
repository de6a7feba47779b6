"""The cluster layout with its cluster capped at 8 CTAs (EP_MAX_CLUSTER_CTAS=8,
and 12, which counts as 8): up to 8 rounds of 32 entries per warp, the
configuration of a device that cannot co-schedule 16 CTAs.  Run in a child
process, since the cap is read once per process; the child compares every
layout array with the oracle."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np
    import torch
    import workloads
    from tests import gpu_harness as gh
    W = workloads.Workload
    cases = [
        workloads.CONFIGS["qwen3_30b_a3b_decode"],   # 2048 entries: 8 CTAs, 1 round
        workloads.CONFIGS["dsv3_decode"],            # 8192 entries: 8 CTAs, 4 rounds
        W("cap8_16000", T=2000, H=256, E=64, K=8, routing="softmax", layout="contig",
          quant="fp8_ue8m0", align=128, R=4, seed=91),   # 8 CTAs, 8 rounds
        W("cap8_masked_over", T=1500, H=128, E=40, K=8, routing="zipf", layout="masked",
          quant="fp8_f32", cap=200, seed=92),      # capacity overflow, 8 rounds
    ]
    for w in cases:
        case = gh.make_case(w)
        g = gh.run_gpu(w, case)
        ref = gh.check_layout(w, case, g)
        gh.check_dispatch(w, case, g, ref)
        assert gh.check_combine(w, case, g, ref) == 1.0
        print("ok", w.name, ref["status"])
""")


@pytest.mark.parametrize("cap", ["8", "12"])
def test_cluster_capped_at_8_ctas_matches_oracle(cap):
    env = dict(os.environ, EP_MAX_CLUSTER_CTAS=cap)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 4
