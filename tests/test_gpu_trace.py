"""EP_NVTX=1 wraps every C-ABI call in an NVTX range (off by default): in a
child process with it set, a layout, dispatch and combine still match the
oracle (without a tool attached the ranges do nothing)."""
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
    import workloads
    from tests import gpu_harness as gh
    for w in (workloads.CONFIGS["qwen3_30b_a3b_decode"],
              workloads.CONFIGS["dsv3_prefill"].with_(T=3000, name="dsv3_prefill_T3000")):
        case = gh.make_case(w)
        g = gh.run_gpu(w, case)
        ref = gh.check_layout(w, case, g)
        gh.check_dispatch(w, case, g, ref)
        assert gh.check_combine(w, case, g, ref) == 1.0
        print("ok", w.name)
""")


def test_nvtx_ranges_change_nothing():
    env = dict(os.environ, EP_NVTX="1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 2
