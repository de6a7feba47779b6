"""Run one entry point on one workload a few times, for profiling.

    python -m combine_expert_histogram_gb300.profile_cases <case> [--reps N]

Cases (seeded synthetic inputs of the named workload, built on the device):

  layout_<workload>    ep_layout (masked layouts with row_src, contiguous otherwise)
  dispatch_<workload>  ep_dispatch in the workload's quantisation mode
  combine_<workload>   ep_combine of bf16 expert outputs
  repack_<workload>    ep_masked_repack of the workload's contiguous dispatch
                       into its masked slab

Every call of the case runs once untimed before the --reps profiled ones, so
that a profiler can skip it (``ncu -s``); the launches of one rep are the
entry point's kernels only.  Nothing is timed or checked here.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np


def main(argv=None) -> int:
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch

    import workloads
    from combine_expert_histogram_gb300 import binding as ep

    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    op, _, name = args.case.partition("_")
    if name not in workloads.CONFIGS or op not in ("layout", "dispatch", "combine", "repack"):
        ap.error(f"unknown case {args.case}")
    w = workloads.CONFIGS[name]
    dev = torch.device("cuda", 0)
    idx, wts, x = workloads.make_inputs(w)
    idx_d = torch.from_numpy(idx).to(dev)
    w_d = torch.from_numpy(wts).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    if op == "repack":
        if w.layout != "masked":
            ap.error("repack cases need a masked workload (its capacity sizes the slab)")
        L = ep.ep_layout(idx_d, w.E, kind="contig", align=128)
        rows, sc, _ = ep.ep_dispatch(L, x_d, w.quant)
        cap = w.cap
        slab = torch.empty((w.E * cap, w.H), dtype=rows.dtype, device=dev)
        slab_sc = None if sc is None else torch.empty((w.E * cap, sc.shape[-1]), dtype=sc.dtype,
                                                      device=dev)
        mm = torch.empty(w.E, dtype=torch.int32, device=dev)
        call = lambda: ep.ep_masked_repack(L, rows, sc, w.quant, cap, slab=slab,
                                           slab_scales=slab_sc, masked_m=mm)
    else:
        L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap,
                          num_ranks=w.R, device=dev)
        ep.ep_layout(idx_d, w.E, out=L)
        if op == "layout":
            call = lambda: ep.ep_layout(idx_d, w.E, out=L)
        elif op == "dispatch":
            rows_t = torch.empty((L.rows_capacity, w.H), device=dev,
                                 dtype=torch.bfloat16 if w.quant == "none" else torch.uint8)
            sc = None if w.quant == "none" else ep.scale_buffer(L, w.H, w.quant, device=dev)
            call = lambda: ep.ep_dispatch(L, x_d, w.quant, out_rows=rows_t, out_scales=sc)
        else:
            y = workloads.make_expert_outputs(L.rows_capacity, w.H, seed=7, device=dev)
            out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
            call = lambda: ep.ep_combine(L, y, w_d, out=out)
    call()
    torch.cuda.synchronize()
    for _ in range(args.reps):
        call()
    torch.cuda.synchronize()
    L.check_status()
    return 0


if __name__ == "__main__":
    sys.exit(main())
