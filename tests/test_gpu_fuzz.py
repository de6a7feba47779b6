"""Seeded random shapes through layout -> dispatch -> combine, against the oracle.

Each case draws T (including both sides of the dispatch kernels' two tokens
per SM boundary), K, E, H (up to the 32768 limit), the quantisation mode, the
layout kind, the alignment or capacity (small capacities overflow on purpose)
and ids with -1 entries and repeated experts; layout, dispatched rows and scales must be
bit-exact, combine within 1 bf16 ulp (expected bit-exact).
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

QUANTS = ["none", "fp8_f32", "fp8_ue8m0", "mxfp8"]


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.choice([0, 1, 7, 100, 303, 304, 305, 609, 777, 1024, 1025, 2500, 9000]))
    E = int(rng.choice([1, 3, 8, 40, 128, 256, 361, 1000, 1024]))
    K = int(rng.integers(1, min(32, max(E, 1)) + 1))
    quant = QUANTS[seed % len(QUANTS)]
    if quant != "none":
        H = int(rng.choice([128, 384, 640, 2048, 4096, 6144, 7168, 9216, 16384, 32768]))
    else:
        H = int(rng.choice([8, 136, 264, 1024, 3072, 7168, 16384, 32768]))
    if H >= 16384:
        T = min(T, 1025)  # keeps the host-side inputs small
    layout = "masked" if rng.random() < 0.4 else "contig"
    align = int(rng.choice([1, 2, 16, 64, 128]))
    cap = int(rng.integers(1, max(2, (T * K) // max(E, 1) * 2 + 2)))
    R = int(rng.choice([r for r in (1, 2, 4, 8) if E % r == 0]))
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    w = workloads.Workload(f"fuzz{seed}", T=T, H=H, E=E, K=K, routing="softmax", layout=layout,
                           quant=quant, align=align, cap=cap, R=R, seed=seed)
    return w, idx, rng


@pytest.mark.parametrize("seed", range(48))
def test_fuzz_parity(seed):
    w, idx, rng = _case(seed)
    wts = rng.random(idx.shape).astype(np.float32)
    x = workloads.make_x(w, rng)
    case = dict(idx=idx, w=wts, x=x, idx_d=torch.from_numpy(idx).cuda(),
                w_d=torch.from_numpy(wts).cuda(),
                x_d=torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref, sample_tokens=512)
    gh.check_combine(w, case, g, ref, sample_tokens=512)
