"""Benchmark: MoE token dispatch + combine on GB300 at the DeepSeek-V3 prefill shape.

One step = ep_layout + ep_dispatch (bf16 -> FP8-E4M3, 1x128 fp32 scales, into
the 128-row-aligned per-expert-contiguous layout) + ep_combine (top-8 weighted
reduction of bf16 expert outputs), for T=16384 tokens, H=7168, E=256, top-8
grouped-sigmoid routing.  Inputs are seeded synthetic data resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  N > 1 (under torchrun) runs independent replicas, one per
GPU, with no collective on the data path ("weak" scaling); a barrier and the
max over ranks bracket the timed region.  ``--impl reference`` times the CPU
oracle on the host cores instead (rank 0 only), on token samples of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (fraction of GB300 peak)"
WORKLOAD = "dsv3_prefill"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "combine_dsv3_prefill_traffic.txt")
# Whole-model serving throughput on 8 GPUs that SGLang PR "[Feature] Add
# DeepEPv2 (ElasticBuffer) MoE A2A backend" reports in its representative
# back-to-back serving results (B200 x8, dynamic blockwise FP8 experts), for
# the DeepEP V2 backend and legacy DeepEP.  Context only: a whole serving
# stack on 8 GPUs, not a single-GPU dispatch / combine figure.
PAGES_CONTEXT = {
    "what": "pages' whole-model serving throughput, 8 GPUs (B200 x8 per the page); "
            "context only, not comparable with this single-GPU kernel metric",
    "decode_tok_s": {"deepep_v2": 8429, "legacy_deepep": 8675},
    "prefill_in_tok_s": {"deepep_v2": 32447, "legacy_deepep": 31533},
}
COMBINE_SRC = os.path.join(ROOT, "combine_expert_histogram_gb300", "csrc", "combine.cu")


# ----------------------------------------------------------- algorithmic bytes
def algorithmic_bytes(w: workloads.Workload) -> dict:
    """Bytes the method must move per launch (padding and empty slots excluded)."""
    T, H, K = w.T, w.H, w.K
    G = H // 128
    row = {"none": 2 * H, "fp8_f32": H + 4 * G, "fp8_ue8m0": H + 4 * ((G + 3) // 4),
           "mxfp8": H + H // 32}[w.quant]
    return dict(
        layout=T * (4 * K + 4 * K + 4 * K),               # idx read, dst_row + row_src written
        dispatch=T * (2 * H + 4 * K + K * row),           # x read, dst_row read, K rows written
        combine=T * (K * 2 * H + 4 * K + 4 * K + 2 * H),  # K rows + w + dst_row read, out written
    )


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in d and d[k]:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def combine_traffic():
    """DRAM bytes per combine launch from the committed ncu summary, if it was
    taken on the current combine.cu (else None)."""
    try:
        src_hash = hashlib.sha256(open(COMBINE_SRC, "rb").read()).hexdigest()[:16]
        kv = {}
        for line in open(TRAFFIC_FILE):
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
        if kv.get("combine_cu_sha256_16") == src_hash:
            return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        pass
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.lines = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                    "-lms", "25"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t_start, t_end, strict=False):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                sm = float(f[2].split()[0])
                smax = float(f[3].split()[0])
            except (ValueError, IndexError):
                continue
            reasons = [n for n, v in zip(("hw_slowdown", "hw_thermal_slowdown",
                                          "sw_thermal_slowdown", "sw_power_cap"), f[6:10])
                       if v.lower().startswith("active")]
            rows.append((ts, sm, smax, reasons))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inwin = [r for r in rows if t_start - 0.025 <= r[0] <= t_end + 0.025]
        window = "timed"
        if strict:
            return {"samples": len(inwin)}
        if not inwin:
            inwin, window = rows, "warmup+timed"
        reasons = sorted({x for r in inwin for x in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in inwin),
                "sm_max_mhz": max(r[2] for r in inwin), "reasons": reasons,
                "samples": len(inwin), "window": window}


def bench_config(w, world: int) -> dict:
    """The workload description both arms print."""
    rows = w.T * w.K + min(w.E, w.T * w.K) * (w.align - 1)
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "K": w.K,
            "routing": {"softmax": "softmax top-k, renormalised",
                        "grouped_sigmoid": "grouped sigmoid + N(0,0.1) bias, "
                                           f"{w.n_group} groups / top-{w.topk_group}",
                        "zipf": "Zipf(1.2) without replacement"}[w.routing],
            "layout": ("expert-contiguous, %d-row aligned" % w.align) if w.layout == "contig"
                      else "masked [E, %d, H]" % w.cap,
            "quant": w.quant,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": (f"inputs larger than L2: x {w.T * w.H * 2 / 1e6:.0f} MB, "
                   f"y {rows * w.H * 2 / 1e9:.2f} GB (L2 129 MB); no flush")}


# ------------------------------------------------------------ replicas
def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank number over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, steps: int, world: int, max_elapsed_ms: float):
    """Whole-job throughput: tokens of all replicas / the slowest rank's time."""
    return tokens_per_rank * steps * world / (max_elapsed_ms * 1e-3)


# ------------------------------------------------------------ CPU baseline
def oracle_tokens_per_s(w, idx, wts, x, y_host, n_tokens):
    """Run the oracle's layout + dispatch + combine on the first n_tokens tokens;
    returns (tokens/s of the whole pass, seconds, seconds per part)."""
    import oracle
    orc = oracle.default()
    sub_idx = np.ascontiguousarray(idx[:n_tokens])
    sub_w = np.ascontiguousarray(wts[:n_tokens])
    sub_x = np.ascontiguousarray(x[:n_tokens])
    t0 = time.perf_counter()
    L = orc.layout(sub_idx, w.E, w.layout, align=w.align, cap=w.cap, R=w.R)
    t1 = time.perf_counter()
    orc.dispatch(sub_x, L["dst_row"], L["rows"], w.quant)
    t2 = time.perf_counter()
    need = max(L["rows"], 1)
    orc.combine(y_host[:need], sub_w, L["dst_row"], w.H)
    t3 = time.perf_counter()
    parts = {"layout": t1 - t0, "dispatch": t2 - t1, "combine": t3 - t2}
    return n_tokens / (t3 - t0), t3 - t0, parts


def part_rates(w, n_tokens, parts):
    """tokens/s and GB/s of each oracle part on the GPU kernels' algorithmic
    bytes per token (the same counts as the kernels' roofline)."""
    per_tok = {k: v / w.T for k, v in algorithmic_bytes(w).items()}
    out = {}
    for k, dt in parts.items():
        out[k] = {"s": round(dt, 4), "tokens_per_s": round(n_tokens / dt, 1),
                  "GB/s": round(per_tok[k] * n_tokens / dt / 1e9, 3)}
    return out


def y_host_rows(w, rows):
    # oracle-side expert outputs: seeded bf16 N(0,1) rows (host generator)
    import torch
    return workloads.make_expert_outputs(rows, w.H, seed=7, device="cpu").view(
        torch.int16).numpy().view(np.uint16)


def cpu_baseline(w, idx, wts, x, target_s=10.0):
    y_host = y_host_rows(w, 256 * w.K + w.E * w.align)
    rate, dt, _ = oracle_tokens_per_s(w, idx, wts, x, y_host, 256)
    n = int(min(w.T, max(256, rate * target_s)))
    if n > 256:
        y_host = y_host_rows(w, n * w.K + w.E * w.align)
    rate, dt, parts = oracle_tokens_per_s(w, idx, wts, x, y_host, n)
    return {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {n} of {w.T} tokens of {w.name}, one pass of layout + dispatch "
                      f"+ combine, single-threaded C oracle ({dt:.1f} s)",
            **part_rates(w, n, parts)}


def oracle_tokens_per_s_threads(w, idx, wts, x, y_host, n_tokens, threads):
    """The same oracle calls on `threads` host threads: the layout (one serial
    scan) on one thread, then dispatch and combine on disjoint token ranges,
    each range writing its own rows of shared outputs (ctypes releases the GIL
    for the duration of every C call)."""
    import ctypes
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    orc = oracle.default()
    lib = orc.lib
    H, K = w.H, w.K
    sub_idx = np.ascontiguousarray(idx[:n_tokens])
    sub_w = np.ascontiguousarray(wts[:n_tokens])
    sub_x = np.ascontiguousarray(x[:n_tokens])
    at = lambda a, off: ctypes.c_void_p(a.ctypes.data + off)
    b = np.linspace(0, n_tokens, threads + 1).astype(int)
    ranges = [(int(b[i]), int(b[i + 1])) for i in range(threads) if b[i + 1] > b[i]]
    with ThreadPoolExecutor(threads) as pool:
        t0 = time.perf_counter()
        L = orc.layout(sub_idx, w.E, w.layout, align=w.align, cap=w.cap, R=w.R)
        t1 = time.perf_counter()
        rows = max(L["rows"], 1)
        d = np.ascontiguousarray(L["dst_row"], dtype=np.int32)
        if w.quant == "none":
            out, sc = np.zeros((rows, H), np.uint16), None
        else:
            out = np.zeros((rows, H), np.uint8)
            sc = np.zeros((rows, oracle.scale_cols(H, w.quant)),
                          np.float32 if w.quant == "fp8_f32" else np.int32)
        comb = np.zeros((n_tokens, H), np.uint16)

        def disp(r):
            lib.orc_dispatch(at(sub_x, r[0] * H * 2), r[1] - r[0], K, H, oracle.QUANT[w.quant],
                             at(d, r[0] * K * 4), at(out, 0),
                             None if sc is None else at(sc, 0), None, None)

        def combine(r):
            lib.orc_combine(at(y_host, 0), at(sub_w, r[0] * K * 4), at(d, r[0] * K * 4),
                            r[1] - r[0], K, H, at(comb, r[0] * H * 2))

        t2 = time.perf_counter()  # output buffers are allocated outside the parts
        list(pool.map(disp, ranges))
        t3 = time.perf_counter()
        list(pool.map(combine, ranges))
        t4 = time.perf_counter()
    parts = {"layout": t1 - t0, "dispatch": t3 - t2, "combine": t4 - t3}
    total = sum(parts.values())
    return n_tokens / total, total, parts


def cpu_baseline_threads(w, idx, wts, x, reps=3):
    """Token-parallel oracle on every host core: median of `reps` runs (whole
    pass), each part's median reported beside it."""
    threads = os.cpu_count() or 1
    n = w.T
    y_host = y_host_rows(w, n * w.K + w.E * w.align)
    runs = [oracle_tokens_per_s_threads(w, idx, wts, x, y_host, n, threads) for _ in range(reps)]
    rate, dt, _ = sorted(runs, key=lambda r: r[1])[len(runs) // 2]
    parts = {k: float(np.median([r[2][k] for r in runs])) for k in ("layout", "dispatch",
                                                                      "combine")}
    return {"value": rate, "unit": "tokens/s", "cores": threads,
            "kind": "oracle, token-parallel",
            "sample": f"all {n} tokens of {w.name}: layout on one thread, dispatch and combine "
                      f"on {threads} threads over disjoint token ranges; median of {reps} "
                      f"({dt:.2f} s)",
            **part_rates(w, n, parts)}


# ---------------------------------------------------------------- reference
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    idx, wts, x = workloads.make_inputs(w)
    y_host = y_host_rows(w, 256 * w.K + w.E * w.align)
    rate, _, _ = oracle_tokens_per_s(w, idx, wts, x, y_host, 256)
    budget = 60.0  # seconds for the whole --warmup + --steps run
    n = int(max(16, min(w.T, rate * budget / max(1, args.steps + args.warmup))))
    y_host = y_host_rows(w, n * w.K + w.E * w.align)
    for _ in range(args.warmup):
        oracle_tokens_per_s(w, idx, wts, x, y_host, n)
    total_dt = 0.0
    part_dt = {"layout": 0.0, "dispatch": 0.0, "combine": 0.0}
    for _ in range(args.steps):
        _, dt, parts = oracle_tokens_per_s(w, idx, wts, x, y_host, n)
        total_dt += dt
        for k in part_dt:
            part_dt[k] += parts[k]
    value = n * args.steps / total_dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": bench_config(w, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"first {n} of {w.T} tokens per step, one pass of "
                                       "layout + dispatch + combine, single-threaded C oracle",
                             **part_rates(w, n * args.steps, part_dt)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- ours
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from combine_expert_histogram_gb300 import binding as ep
    from combine_expert_histogram_gb300 import build as epbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    if not epbuild.up_to_date() and rank == 0:
        epbuild.build()
    if world > 1:
        dist.barrier()

    # inputs (seeded; each replica gets its own batch)
    wr = w.with_(seed=w.seed + rank)
    idx, wts, x = workloads.make_inputs(wr)
    idx_d = torch.from_numpy(idx).to(dev)
    w_d = torch.from_numpy(wts).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R,
                      device=dev)
    rows = L.rows_capacity
    out_rows = torch.empty((rows, w.H), device=dev,
                           dtype=torch.bfloat16 if w.quant == "none" else torch.uint8)
    out_scales = None
    if w.quant != "none":
        out_scales = torch.empty((rows, ep.ep_scale_cols(w.H, w.quant)), device=dev,
                                 dtype=torch.float32 if w.quant == "fp8_f32" else torch.int32)
    y = workloads.make_expert_outputs(rows, w.H, seed=7 + rank, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    n_layout_kernels = 2 if ep.ep_layout_workspace_bytes(L) > 0 else 1
    launches_per_step = n_layout_kernels + 2

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ep.ep_layout(idx_d, w.E, out=L, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        ep.ep_dispatch(L, x_d, w.quant, out_rows=out_rows, out_scales=out_scales, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        ep.ep_combine(L, y, w_d, out=out, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    L.check_status()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    # The timed steps carry no event between kernels: an event there would
    # also cut the programmatic (overlapped) launch of the next kernel, so the
    # steps run exactly as a caller would run them.
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), dev if world > 1 else None)

    # Per-kernel times, independent of --steps: further steps with an event
    # between every two kernels (each kernel then starts only after the one
    # before it has finished), at least --kernel-reps of them and at least
    # --kernel-seconds of GPU time, median per kernel.  The clock sampler keeps
    # running through these steps, so the clock record covers more than the
    # (possibly short) timed region.
    kreps = max(args.kernel_reps, int(math.ceil(args.kernel_seconds * 1e3 * args.steps
                                                 / max(elapsed_ms, 1e-3))))
    kreps = min(kreps, 20000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(kreps)]
    with torch.cuda.stream(stream):
        for e in evs:
            step(e)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    seg = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in evs])
    ab = algorithmic_bytes(w)
    peak, peak_src = peak_hbm()
    kern = {}
    # the survey's "dispatch" figure: ep_layout + ep_dispatch, per step
    both = seg[:, 0] + seg[:, 1]
    both_us = float(np.median(both)) * 1e3
    kern["layout_plus_dispatch"] = {
        "us": round(both_us, 2), "tokens_per_s": round(w.T / (both_us * 1e-6), 1),
        "GB/s": round((ab["layout"] + ab["dispatch"]) / (both_us * 1e-6) / 1e9, 1),
        "frac_of_peak": round((ab["layout"] + ab["dispatch"]) / (both_us * 1e-6) / 1e9 / peak, 4)}
    for j, name in enumerate(("layout", "dispatch", "combine")):
        ms = float(np.median(seg[:, j]))
        gbs = ab[name] / (ms * 1e-3) / 1e9
        kern[name] = {"us": round(ms * 1e3, 2), "us_mean": round(float(seg[:, j].mean()) * 1e3, 2),
                      "us_p10_p90": [round(float(np.percentile(seg[:, j], q)) * 1e3, 2)
                                     for q in (10, 90)],
                      "launches": int(kreps), "algorithmic_bytes": ab[name],
                      "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}

    # end to end through the public API with pinned host buffers
    # end to end on every rank (each replica has its own host link), slowest rank counts
    e2e = None
    if not args.skip_e2e:
        if world > 1:
            dist.barrier()
        e2e = measure_e2e(ep, w, L, idx, wts, x, y, out_rows, out_scales, dev, stream, args)
        e2e_ms = max_over_ranks(e2e["ms_per_step"], dev if world > 1 else None)
        e2e["ms_per_step"] = e2e_ms
        e2e["value"] = w.T * world / (e2e_ms * 1e-3)

    if rank != 0:
        dist.destroy_process_group()
        return
    value = aggregate_tokens_per_s(w.T, args.steps, world, elapsed_ms)
    dom = max(("dispatch", "combine"), key=lambda k: kern[k]["us"])
    traffic = combine_traffic() if dom == "combine" else None
    achieved = kern[dom]["GB/s"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",
        "formats": "bf16 activations in; E4M3 rows + fp32 1x128 scales out of dispatch; "
                   "bf16 expert outputs in, fp32 accumulation, bf16 out of combine",
        "data": "synthetic",
        "config": bench_config(w, world),
        "step_gbs": round(sum(ab.values()) * args.steps * world / (elapsed_ms * 1e-3) / 1e9, 1),
        "kernels": kern,
        "kernel_events": (f"median over {kreps} further steps with an event between every two "
                          "kernels (none in the timed steps)"),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": ab[dom]},
        "gpu_launches": launches_per_step * args.steps,
    }
    if sampler:
        # the timed steps and the per-kernel timing steps that follow them
        line["clocks"] = sampler.summary(t_wall0, t_wall2)
        line["clocks"]["window"] = "timed steps + per-kernel timing steps"
        line["clocks"]["samples_timed_only"] = sampler.summary(t_wall0, t_wall1, strict=True)["samples"]
    if e2e:
        line["e2e"] = e2e
    sections = set(args.sections.split(",")) if args.sections else set()
    if args.skip_decode:
        sections = set()
    if "variants" in sections:
        line["dispatch_variants"] = measure_dispatch_variants(ep, w, L, x_d, dev)
    if "decode" in sections:
        line["decode"] = measure_decode(ep, dev)
    if "rank" in sections:
        line["rank_dedup"] = measure_rank_dedup(ep, dev)
    if "router" in sections:
        line["router"] = measure_router(ep, dev)
    if "skewed" in sections:
        line["skewed_zipf"] = measure_skewed(ep, dev, peak)
    line["context"] = PAGES_CONTEXT
    if not args.skip_cpu and world == 1:  # the CPU baseline is an N=1 figure
        line["cpu_baseline"] = cpu_baseline(w, idx, wts, x)
        line["cpu_baseline_threads"] = cpu_baseline_threads(w, idx, wts, x)
    if rank == 0:
        print_table(line)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def print_table(line, out=None):
    """A human-readable summary of the bench line on stderr (stdout keeps the
    single JSON line): workload, per-kernel time, tokens/s, GB/s and fraction
    of the HBM peak, the decode steps and the CPU oracle."""
    out = out or sys.stderr
    c = line.get("config", {})
    rows = [("step (layout + dispatch + combine)", line.get("ms_per_step", 0) * 1e3,
             line.get("value"), line.get("step_gbs"), None)]
    T = c.get("T") or 0
    for name, k in line.get("kernels", {}).items():
        tps = k.get("tokens_per_s") or (T / (k["us"] * 1e-6) if k.get("us") else None)
        rows.append((name, k.get("us"), tps, k.get("GB/s"), k.get("frac_of_peak")))

    def fmt(v, f):
        width = int("".join(ch for ch in f.split(".")[0] if ch.isdigit()) or 0)
        return format("-", f">{width}") if v is None else format(v, f)
    print(f"{c.get('workload', '?')}: T={c.get('T')} H={c.get('H')} E={c.get('E')} K={c.get('K')} "
          f"quant={c.get('quant')}, peak {line.get('roofline', {}).get('peak')} GB/s "
          f"({line.get('roofline', {}).get('peak_source')})", file=out)
    print(f"  {'':36s} {'us':>9s} {'tokens/s':>12s} {'GB/s':>8s} {'of peak':>8s}", file=out)
    for name, us, tps, gbs, frac in rows:
        print(f"  {name:36s} {fmt(us, '9.2f')} {fmt(tps, '12.4g')} {fmt(gbs, '8.1f')} "
              f"{fmt(frac, '8.3f')}", file=out)
    for name, d in line.get("decode", {}).items():
        print(f"  decode {name}: step {d['step_us_graph']} us from CUDA graphs "
              f"(from logits {d.get('from_logits', {}).get('step_us_graph')} us); layout "
              f"{d['warm_graph_us']['layout']} us warm", file=out)
    for key in ("cpu_baseline", "cpu_baseline_threads"):
        b = line.get(key)
        if b:
            print(f"  CPU oracle ({b['cores']} core{'s' if b['cores'] != 1 else ''}): "
                  f"{b['value']:.4g} tokens/s", file=out)
    e = line.get("e2e")
    if e:
        print(f"  end to end from pinned host memory: {e['value']:.4g} tokens/s", file=out)


def graph_time_us(fns, stream, reps=50, flush=None, trials=5):
    """GPU time of one pass of `fns` (callables launching on `stream`), from a
    CUDA graph holding `reps` passes back to back: no host launch overhead
    enters.  One untimed replay warms up, then the median over `trials` timed
    replays is divided by `reps`.  With `flush` (a callable writing 2x L2),
    each pass starts from a flushed L2 and a flush-only graph's time is
    subtracted."""
    import torch

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                body()
        return g

    def run(g):
        g.replay()
        torch.cuda.synchronize()
        events = []
        for _ in range(trials):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            events.append((a, b))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in events])) * 1e3 / reps

    def body():
        if flush is not None:
            flush()
        for f in fns:
            f()

    with torch.cuda.stream(stream):
        t = run(capture(body))
        if flush is not None:
            t -= run(capture(flush))
    return t


def measure_decode(ep, dev, reps=50):
    """Decode shapes (masked layouts), timed from CUDA graphs: the whole step
    back to back (warm L2), each kernel from a flushed L2, and the masked
    repack on its own."""
    import torch
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)  # 2x L2
    res = {}
    for name in ("qwen3_30b_a3b_decode", "dsv3_decode"):
        w = workloads.CONFIGS[name]
        idx, wts, x = workloads.make_inputs(w)
        idx_d = torch.from_numpy(idx).to(dev)
        w_d = torch.from_numpy(wts).to(dev)
        x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        L = ep.new_layout(w.T, w.K, w.E, "masked", capacity=w.cap, device=dev)
        rows = L.rows_capacity
        out_rows = torch.empty((rows, w.H), dtype=torch.uint8, device=dev)
        sc = ep.scale_buffer(L, w.H, w.quant, device=dev)
        y = workloads.make_expert_outputs(rows, w.H, seed=3, device=dev)
        out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        s = torch.cuda.Stream(device=dev)
        lay = lambda: ep.ep_layout(idx_d, w.E, out=L, stream=s)
        dis = lambda: ep.ep_dispatch(L, x_d, w.quant, out_rows=out_rows, out_scales=sc, stream=s)
        com = lambda: ep.ep_combine(L, y, w_d, out=out, stream=s)
        fus = lambda: ep.ep_layout_dispatch(idx_d, L, x_d, w.quant, out_rows=out_rows,
                                            out_scales=sc, stream=s)
        flush = lambda: flush_buf.fill_(1)
        with torch.cuda.stream(s):
            for _ in range(3):
                lay(), dis(), com(), fus(), com()
        torch.cuda.synchronize()
        step_us = graph_time_us([lay, dis, com], s, reps)
        one_call_us = graph_time_us([fus, com], s, reps)  # ep_layout_dispatch + ep_combine
        # the same step with a layout that has no row_src (the masked decode
        # path reads only dst_row and the counts)
        Ln = ep.new_layout(w.T, w.K, w.E, "masked", capacity=w.cap, device=dev, with_row_src=False)
        lay_n = lambda: ep.ep_layout(idx_d, w.E, out=Ln, stream=s)
        dis_n = lambda: ep.ep_dispatch(Ln, x_d, w.quant, out_rows=out_rows, out_scales=sc, stream=s)
        com_n = lambda: ep.ep_combine(Ln, y, w_d, out=out, stream=s)
        with torch.cuda.stream(s):
            lay_n(), dis_n(), com_n()
        torch.cuda.synchronize()
        step_n_us = graph_time_us([lay_n, dis_n, com_n], s, reps)
        lay_n_warm = graph_time_us([lay_n], s, reps)
        lay_n_cold = graph_time_us([lay_n], s, reps, flush=flush)
        # the step from router logits (fp32 [T, E], seeded N(0, 1), bias N(0, 0.1)):
        # ep_route_topk, then the three calls on its topk_idx / topk_w
        gen = torch.Generator(device=dev)
        gen.manual_seed(17)
        lg = torch.randn((w.T, w.E), generator=gen, device=dev, dtype=torch.float32)
        bias = 0.1 * torch.randn(w.E, generator=gen, device=dev, dtype=torch.float32)
        idx_r = torch.empty((w.T, w.K), dtype=torch.int32, device=dev)
        w_r = torch.empty((w.T, w.K), dtype=torch.float32, device=dev)
        if w.routing == "softmax":
            rte = lambda: ep.ep_route_topk(lg, w.K, "softmax", topk_idx=idx_r, topk_w=w_r,
                                           stream=s)
        else:
            rte = lambda: ep.ep_route_topk(lg, w.K, "grouped_sigmoid", bias=bias,
                                           n_group=w.n_group, topk_group=w.topk_group,
                                           topk_idx=idx_r, topk_w=w_r, stream=s)
        lay_r = lambda: ep.ep_layout(idx_r, w.E, out=L, stream=s)
        com_r = lambda: ep.ep_combine(L, y, w_r, out=out, stream=s)
        with torch.cuda.stream(s):
            rte(), lay_r(), dis(), com_r()
        torch.cuda.synchronize()
        step_r_us = graph_time_us([rte, lay_r, dis, com_r], s, reps)
        rte_us = graph_time_us([rte], s, reps)
        cold = {k: graph_time_us([f], s, reps, flush=flush)
                for k, f in (("layout", lay), ("dispatch", dis), ("combine", com))}
        warm = {k: graph_time_us([f], s, reps)
                for k, f in (("layout", lay), ("dispatch", dis), ("combine", com))}
        ab = algorithmic_bytes(w)
        # masked repack from a contiguous layout (same routing)
        Lc = ep.new_layout(w.T, w.K, w.E, "contig", align=128, device=dev)
        ep.ep_layout(idx_d, w.E, out=Lc)
        rows_c, sc_c, _ = ep.ep_dispatch(Lc, x_d, w.quant)
        slab = torch.empty_like(out_rows)
        slab_sc = torch.empty_like(sc)
        mm = torch.empty(w.E, dtype=torch.int32, device=dev)
        rep = lambda: ep.ep_masked_repack(Lc, rows_c, sc_c, w.quant, w.cap, slab=slab,
                                          slab_scales=slab_sc, masked_m=mm, stream=s)
        with torch.cuda.stream(s):
            rep()
        torch.cuda.synchronize()
        rep_us = graph_time_us([rep], s, reps, flush=flush)
        rep_bytes = 2 * w.T * w.K * (w.H + 4 * sc.shape[-1])  # valid rows read + written
        res[name] = {
            "T": w.T, "H": w.H, "E": w.E, "K": w.K, "cap": w.cap, "quant": w.quant,
            "step_us_graph": round(step_us, 2),
            "tokens_per_s": round(w.T / (step_us * 1e-6), 1),
            "step_us_graph_ep_layout_dispatch": round(one_call_us, 2),
            "from_logits": {"step_us_graph": round(step_r_us, 2),
                            "router_us_graph": round(rte_us, 2),
                            "what": "ep_route_topk + ep_layout + ep_dispatch + ep_combine"},
            "without_row_src": {"step_us_graph": round(step_n_us, 2),
                                "layout_warm_us": round(lay_n_warm, 2),
                                "layout_l2_flushed_us": round(lay_n_cold, 2)},
            "l2_flushed_us": {k: round(v, 2) for k, v in cold.items()},
            "warm_graph_us": {k: round(v, 2) for k, v in warm.items()},
            "dispatch_GBps_flushed": round(ab["dispatch"] / (cold["dispatch"] * 1e-6) / 1e9, 1),
            "combine_GBps_flushed": round(ab["combine"] / (cold["combine"] * 1e-6) / 1e9, 1),
            "masked_repack_us_flushed": round(rep_us, 2),
            "masked_repack_GBps": round(rep_bytes / (rep_us * 1e-6) / 1e9, 1),
        }
        del y, out_rows, slab, rows_c
        torch.cuda.empty_cache()
    return res


def measure_skewed(ep, dev, peak, reps=100):
    """The skewed-load workload (T=8192, H=4096, E=128, top-8 Zipf(1.2) experts,
    Dirichlet weights; 8 logical ranks of 16 experts; bf16 rows): layout,
    dispatch and combine each timed with CUDA events in steps of the three
    calls (an event between every two kernels), median over `reps` steps.
    Between two steps the combine streams 0.6 GB through L2, which evicts the
    67 MB of x that the next dispatch reads."""
    import torch
    w = workloads.CONFIGS["skewed_zipf"]
    idx, wts, x = workloads.make_inputs(w)
    idx_d = torch.from_numpy(idx).to(dev)
    w_d = torch.from_numpy(wts).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, num_ranks=w.R, device=dev)
    rows = L.rows_capacity
    out_rows = torch.empty((rows, w.H), dtype=torch.bfloat16, device=dev)
    y = workloads.make_expert_outputs(rows, w.H, seed=7, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)

    def step(e):
        e[0].record(s)
        ep.ep_layout(idx_d, w.E, out=L, stream=s)
        e[1].record(s)
        ep.ep_dispatch(L, x_d, w.quant, out_rows=out_rows, stream=s)
        e[2].record(s)
        ep.ep_combine(L, y, w_d, out=out, stream=s)
        e[3].record(s)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps + 5)]
    with torch.cuda.stream(s):
        for e in evs:
            step(e)
    torch.cuda.synchronize()
    L.check_status()
    seg = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in evs[5:]])
    ab = algorithmic_bytes(w)
    res = {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "K": w.K, "ranks": w.R,
           "quant": "bf16 rows", "steps_timed": reps,
           "algorithmic_bytes_per_token": {k: ab[k] // w.T for k in ("dispatch", "combine")}}
    for j, name in enumerate(("layout", "dispatch", "combine")):
        us = float(np.median(seg[:, j])) * 1e3
        gbs = ab[name] / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 2), "tokens_per_s": round(w.T / (us * 1e-6), 1),
                     "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
    rr = L.rank_rows.cpu().numpy().astype(int)
    cnt = L.expert_count.cpu().numpy().astype(int)
    off = L.expert_offset.cpu().numpy().astype(int)
    per = w.E // w.R
    res["rank_rows"] = rr.tolist()
    res["rank_rows_padded"] = [int(off[(r + 1) * per] - off[r * per]) for r in range(w.R)]
    res["hot_rank_share"] = round(float(rr.max() / max(rr.sum(), 1)), 4)
    res["hottest_expert_rows"] = int(cnt.max())
    del out_rows, y
    torch.cuda.empty_cache()
    return res


def measure_dispatch_variants(ep, w, L, x_d, dev, reps=20):
    """ep_dispatch alone in every quantisation mode on the bench workload's layout
    (inputs larger than L2); algorithmic bytes as in algorithmic_bytes()."""
    import torch
    res = {}
    rows = L.rows_capacity
    for quant in ("fp8_f32", "fp8_ue8m0", "fp8_ue8m0_mn", "mxfp8", "none"):
        out_rows = torch.empty((rows, w.H), device=dev,
                               dtype=torch.bfloat16 if quant == "none" else torch.uint8)
        sc = ep.scale_buffer(L, w.H, quant, device=dev)
        for _ in range(3):
            ep.ep_dispatch(L, x_d, quant, out_rows=out_rows, out_scales=sc)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            ep.ep_dispatch(L, x_d, quant, out_rows=out_rows, out_scales=sc)
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        nbytes = algorithmic_bytes(w.with_(quant=quant.replace("_mn", "")))["dispatch"]
        res[quant] = {"us": round(us, 2), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                      "tokens_per_s": round(w.T / (us * 1e-6), 1)}
        del out_rows, sc
    return res


def measure_router(ep, dev, reps=20):
    """ep_route_topk at the two router families' bench shapes (fp32 logits),
    timed from a CUDA graph of back-to-back calls."""
    import torch
    res = {}
    for name, T, E, K, mode, G, TG in (("dsv3_prefill", 16384, 256, 8, "grouped_sigmoid", 8, 4),
                                       ("dsv3_decode", 1024, 256, 8, "grouped_sigmoid", 8, 4),
                                       ("qwen3_30b_a3b_decode", 256, 128, 8, "softmax", 1, 1)):
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        lg = torch.randn((T, E), generator=g, device=dev, dtype=torch.float32)
        bias = torch.randn(E, generator=g, device=dev, dtype=torch.float32) * 0.1
        idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        wts = torch.empty((T, K), dtype=torch.float32, device=dev)
        s = torch.cuda.Stream(device=dev)

        def run():
            ep.ep_route_topk(lg, K, mode, bias=bias, n_group=G, topk_group=TG, topk_idx=idx,
                             topk_w=wts, stream=s)

        with torch.cuda.stream(s):
            for _ in range(3):
                run()
        torch.cuda.synchronize()
        us = graph_time_us([run], s, reps)
        nbytes = T * E * 4 + E * 4 + T * K * 8
        res[name] = {"mode": mode, "T": T, "E": E, "K": K, "us": round(us, 2),
                     "tokens_per_s": round(T / (us * 1e-6), 1),
                     "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1)}
    return res


def measure_rank_dedup(ep, dev, reps=10):
    """Per-rank deduplicated sending at the Zipf workload (8 logical ranks):
    rank layout + dispatch into the send buffer + local expand, beside the
    direct dispatch of the same tokens (CUDA-graph timing)."""
    import torch
    w = workloads.CONFIGS["skewed_zipf"]
    idx, wts, x = workloads.make_inputs(w)
    idx_d = torch.from_numpy(idx).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    L = ep.ep_layout(idx_d, w.E, align=w.align, num_ranks=w.R)
    RL, rank_idx = ep.ep_rank_layout(idx_d, w.E, w.R)
    send_rows, _, _ = ep.ep_dispatch(RL, x_d, w.quant)
    out_rows, _ = ep.ep_rank_expand(RL, L, idx_d, w.quant, send_rows, None)
    direct, _, _ = ep.ep_dispatch(L, x_d, w.quant)
    torch.cuda.synchronize()
    send_n = int(RL.expert_offset[-1].item())

    s = torch.cuda.Stream(device=dev)

    def timed(fn):
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        return graph_time_us([fn], s, reps)

    t_rl = timed(lambda: ep.ep_rank_layout(idx_d, w.E, w.R, out=RL, rank_idx=rank_idx, stream=s))
    t_send = timed(lambda: ep.ep_dispatch(RL, x_d, w.quant, out_rows=send_rows, stream=s))
    t_exp = timed(lambda: ep.ep_rank_expand(RL, L, idx_d, w.quant, send_rows, None,
                                            out_rows=out_rows, stream=s))
    t_direct = timed(lambda: ep.ep_dispatch(L, x_d, w.quant, out_rows=direct, stream=s))
    row = 2 * w.H
    send_bytes = w.T * row + send_n * row + w.T * w.K * 4
    exp_bytes = send_n * row + w.T * w.K * row + 2 * w.T * w.K * 4
    return {"workload": w.name, "ranks": w.R, "send_rows": send_n,
            "rows_per_token": round(send_n / w.T, 3),
            "rank_layout_us": round(t_rl, 2),
            "send_dispatch_us": round(t_send, 2),
            "send_dispatch_GBps": round(send_bytes / (t_send * 1e-6) / 1e9, 1),
            "expand_us": round(t_exp, 2),
            "expand_GBps": round(exp_bytes / (t_exp * 1e-6) / 1e9, 1),
            "direct_dispatch_us": round(t_direct, 2)}


def numa_placement(t) -> dict:
    """NUMA nodes of the host, and the nodes holding the pages of pinned tensor t
    (from /proc/self/numa_maps; Linux only)."""
    import glob
    nodes = {}
    for n in sorted(glob.glob("/sys/devices/system/node/node[0-9]*")):
        try:
            nodes[os.path.basename(n)] = open(n + "/cpulist").read().strip()
        except OSError:
            pass
    lo, hi = t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()
    pages = {}
    try:
        for line in open("/proc/self/numa_maps"):
            f = line.split()
            if lo <= int(f[0], 16) < hi:
                for tok in f:
                    if tok[:1] == "N" and "=" in tok:
                        k, v = tok.split("=")
                        pages[k] = pages.get(k, 0) + int(v)
    except (OSError, ValueError):
        pass
    return {"host_nodes_cpus": nodes, "pinned_pages_by_node": pages}


def link_rates(h, d, stream) -> dict:
    """Host->device, device->host and both at once (two streams), GB/s, on
    the pinned host tensor h and a device tensor d of the same bytes."""
    import torch
    other = torch.cuda.Stream(device=d.device)
    hb = torch.empty_like(h, pin_memory=True)
    db = torch.empty_like(d)
    nbytes = h.numel() * h.element_size()

    def timed(fn):
        best = None
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return best

    def up():
        with torch.cuda.stream(stream):
            d.copy_(h, non_blocking=True)

    def down():
        with torch.cuda.stream(stream):
            hb.copy_(db, non_blocking=True)

    def both():
        up()
        with torch.cuda.stream(other):
            hb.copy_(db, non_blocking=True)

    tb = timed(both)
    return {"h2d_GBps": round(nbytes / timed(up) / 1e9, 1),
            "d2h_GBps": round(nbytes / timed(down) / 1e9, 1),
            "both_at_once_GBps_each": round(nbytes / tb / 1e9, 1),
            "bytes": nbytes, "method": "one cudaMemcpyAsync per direction from pinned memory, "
                                        "best of 3; both: two streams"}


def measure_e2e(ep, w, L, idx, wts, x, y_dev, out_rows, out_scales, dev, stream, args):
    """Same metric through the public API with inputs in pinned host memory:
    every step copies x, topk_idx, topk_w and the expert outputs y host->device,
    runs layout + dispatch + combine and copies the combined output (and the
    expert histogram) back.  Steps are pipelined the way a serving loop would
    run them: inputs are double-buffered on the device, so step i+1's inputs
    travel host->device while step i computes and its output travels back.
    Uploads and downloads together are bound by the host link (about 211 GB/s
    measured for both directions combined)."""
    import torch
    pin = dict(pin_memory=True)
    h_idx = torch.from_numpy(idx).pin_memory()
    h_w = torch.from_numpy(wts).pin_memory()
    h_x = torch.from_numpy(x.view(np.int16)).pin_memory()
    h_y = torch.empty(y_dev.shape, dtype=torch.int16, **pin)
    h_y.copy_(y_dev.view(torch.int16))
    h_out = [torch.empty((w.T, w.H), dtype=torch.int16, **pin) for _ in range(2)]
    h_cnt = [torch.empty(w.E, dtype=torch.int32, **pin) for _ in range(2)]
    bufs = [dict(idx=torch.empty_like(h_idx, device=dev), w=torch.empty_like(h_w, device=dev),
                 x=torch.empty(h_x.shape, dtype=torch.int16, device=dev),
                 y=torch.empty(h_y.shape, dtype=torch.int16, device=dev),
                 out=torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev),
                 cnt=torch.empty(w.E, dtype=torch.int32, device=dev))
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_idx, h_w, h_x, h_y))
    d2h = h_out[0].numel() * 2 + h_cnt[0].numel() * 4
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {}

    def step(i):
        b = bufs[i % 2]
        if i >= 2:  # the compute of step i-2 has read this buffer set
            up.wait_event(ev[("done", i - 2)])
        with torch.cuda.stream(up):
            b["idx"].copy_(h_idx, non_blocking=True)
            b["w"].copy_(h_w, non_blocking=True)
            b["x"].copy_(h_x, non_blocking=True)
            b["y"].copy_(h_y, non_blocking=True)
            ev[("in", i)] = torch.cuda.Event()
            ev[("in", i)].record(up)
        stream.wait_event(ev[("in", i)])
        if i >= 2:  # the output of step i-2 has left this buffer set
            stream.wait_event(ev[("out", i - 2)])
        with torch.cuda.stream(stream):
            ep.ep_layout(b["idx"], w.E, out=L, stream=stream)
            ep.ep_dispatch(L, b["x"].view(torch.bfloat16), w.quant, out_rows=out_rows,
                           out_scales=out_scales, stream=stream)
            ep.ep_combine(L, b["y"].view(torch.bfloat16), b["w"], out=b["out"], stream=stream)
            b["cnt"].copy_(L.expert_count, non_blocking=True)
            ev[("done", i)] = torch.cuda.Event()
            ev[("done", i)].record(stream)
        down.wait_event(ev[("done", i)])
        with torch.cuda.stream(down):
            h_out[i % 2].copy_(b["out"].view(torch.int16), non_blocking=True)
            h_cnt[i % 2].copy_(b["cnt"], non_blocking=True)
            ev[("out", i)] = torch.cuda.Event()
            ev[("out", i)].record(down)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    ev.clear()
    n = max(3, min(args.steps, 20))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for i in range(n):
        step(i)
    down.wait_stream(stream)
    t1.record(down)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    link = link_rates(h_x, bufs[0]["x"], up)
    link.update(numa_placement(h_x))
    # one step's four uploads alone (no compute, no downloads), median of 5:
    # the floor of the e2e step on this machine's host link
    b = bufs[0]
    t_up = []
    for _ in range(5):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(up)
        with torch.cuda.stream(up):
            b["idx"].copy_(h_idx, non_blocking=True)
            b["w"].copy_(h_w, non_blocking=True)
            b["x"].copy_(h_x, non_blocking=True)
            b["y"].copy_(h_y, non_blocking=True)
        a1.record(up)
        torch.cuda.synchronize()
        t_up.append(a0.elapsed_time(a1))
    up_ms = float(np.median(t_up))
    link["step_uploads_ms"] = round(up_ms, 2)
    link["step_uploads_GBps"] = round(h2d / (up_ms * 1e-3) / 1e9, 1)
    return {"value": w.T / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "steps": n,
            "pipelined": "double-buffered inputs; copies up, compute, copies down overlap across steps",
            "host_link": link}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle baseline")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the host-buffer e2e leg")
    ap.add_argument("--kernel-reps", type=int, default=100,
                    help="minimum number of per-kernel timing steps after the timed region")
    ap.add_argument("--kernel-seconds", type=float, default=0.5,
                    help="minimum GPU time of the per-kernel timing steps")
    ap.add_argument("--skip-decode", action="store_true",
                    help="omit every extra measurement section (same as --sections '')")
    ap.add_argument("--sections", default="variants,decode,rank,router,skewed",
                    help="extra measurements after the timed steps: variants (dispatch in "
                         "every quantisation mode), decode (masked decode shapes), rank "
                         "(per-rank deduplicated sending), router (ep_route_topk), skewed "
                         "(the Zipf-skewed bf16 workload's layout, dispatch and combine)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (small cases for profiling; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = workloads.CONFIGS[args.workload]
    if args.tokens:
        w = w.with_(T=args.tokens, name=f"{w.name}_T{args.tokens}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
