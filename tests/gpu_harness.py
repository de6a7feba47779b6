"""Run the CUDA path through the C ABI and compare it with the CPU oracle.

Comparisons:
  * layout (counts, offsets, dst_row, row_src, rank_rows, status): bit-exact;
  * dispatched rows and scales (bf16, E4M3 bytes, fp32 / UE8M0 scales):
    bit-exact on every valid row of every token (or of sampled tokens where a
    caller asks for a sample), compared in token chunks, and rows the layout
    leaves empty keep their sentinel bytes;
  * combine output: within 1 bf16 ulp (the two sides use the same summation
    order, so it is expected to be bit-exact; ``exact_fraction`` reports it).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads
from combine_expert_histogram_gb300 import binding as ep

SENTINEL_U8 = 0xA5
SENTINEL_BF16 = -23131  # int16 view of 0xA5A5
# tokens per oracle call when comparing dispatch and combine (bounds host memory:
# 2048 tokens of the DeepSeek-V3 shape are 117 MB of E4M3 rows, 235 MB of y)
CHUNK_TOKENS = 2048


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 ulps, by the ordered-integer distance of the bit patterns."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a) - key(b))


def make_case(w: workloads.Workload, device="cuda"):
    idx, wts, x = workloads.make_inputs(w)
    return dict(idx=idx, w=wts, x=x,
                idx_d=torch.from_numpy(idx).to(device),
                w_d=torch.from_numpy(wts).to(device),
                x_d=torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16))


def run_gpu(w: workloads.Workload, case, with_row_src=True, y_seed=7):
    """layout -> dispatch -> combine on the GPU; returns a dict of device tensors."""
    dev = case["idx_d"].device
    L = ep.ep_layout(case["idx_d"], w.E, kind=w.layout, align=w.align, capacity=w.cap,
                     num_ranks=w.R, with_row_src=with_row_src)
    rows = L.rows_capacity
    H = w.H
    if w.quant == "none":
        out_rows = torch.full((max(rows, 1), H), SENTINEL_BF16, dtype=torch.int16,
                              device=dev).view(torch.bfloat16)
        out_scales = None
    else:
        out_rows = torch.full((max(rows, 1), H), SENTINEL_U8, dtype=torch.uint8, device=dev)
        cols = ep.ep_scale_cols(H, w.quant)
        sdt = torch.float32 if w.quant == "fp8_f32" else torch.int32
        out_scales = torch.zeros((max(rows, 1), cols), dtype=sdt, device=dev)
    row_w = torch.zeros(max(rows, 1), dtype=torch.float32, device=dev)
    ep.ep_dispatch(L, case["x_d"], w.quant, out_rows=out_rows, out_scales=out_scales,
                   topk_w=case["w_d"], row_w=row_w)
    if w.identity_experts:
        assert w.quant == "none"
        y = out_rows
    else:
        y = workloads.make_expert_outputs(max(rows, 1), H, seed=y_seed, device=dev)
    out = ep.ep_combine(L, y, case["w_d"])
    torch.cuda.synchronize()
    return dict(L=L, rows=rows, out_rows=out_rows, out_scales=out_scales, row_w=row_w, y=y,
                out=out)


def check_layout(w, case, g, orc=None):
    orc = orc or oracle.default()
    ref = orc.layout(case["idx"], w.E, w.layout, align=w.align, cap=w.cap, R=w.R)
    L = g["L"]
    T, K = case["idx"].shape
    assert int(L.status.item()) == ref["status"]
    assert np.array_equal(L.expert_count.cpu().numpy(), ref["count"])
    assert np.array_equal(L.expert_offset.cpu().numpy(), ref["offset"])
    if T * K:
        assert np.array_equal(L.dst_row.cpu().numpy()[:T * K].reshape(T, K), ref["dst_row"])
    assert np.array_equal(L.rank_rows.cpu().numpy(), ref["rank_rows"])
    if L.row_src is not None:
        assert np.array_equal(L.row_src.cpu().numpy()[:ref["rows"]], ref["row_src"])
    return ref


def check_dispatch(w, case, g, ref, sample_tokens=None, seed=0, orc=None, check_row_w=True,
                   check_empty=None):
    """Bit-exact rows/scales/row_w; sentinel kept on rows the layout leaves empty.
    Returns the number of tokens whose rows were compared."""
    if check_empty is None:
        check_empty = check_row_w
    orc = orc or oracle.default()
    T, K = case["idx"].shape
    if T == 0:
        return 0
    dst = ref["dst_row"]
    if sample_tokens is None or sample_tokens >= T:
        toks = np.arange(T)
    else:
        rng = np.random.default_rng(seed)
        toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, sample_tokens, replace=False)]))
    # token chunks bound the host memory of the oracle's rows and the copies
    for c0 in range(0, toks.size, CHUNK_TOKENS):
        _check_dispatch_tokens(w, case, g, dst, toks[c0:c0 + CHUNK_TOKENS], orc, check_row_w)
    if not check_empty:
        return int(toks.size)
    # rows no entry maps to keep the sentinel (padding and empty slots)
    rows = ref["rows"]
    used = torch.zeros(max(rows, 1), dtype=torch.bool, device=g["out_rows"].device)
    alld = torch.from_numpy(dst[dst >= 0].astype(np.int64)).to(used.device)
    used[alld] = True
    empty = ~used[:rows]
    if empty.any():
        buf = g["out_rows"][:rows][empty]
        if w.quant == "none":
            assert bool((buf.view(torch.int16) == SENTINEL_BF16).all())
        else:
            assert bool((buf == SENTINEL_U8).all())
    return int(toks.size)


def _check_dispatch_tokens(w, case, g, dst, toks, orc, check_row_w):
    """Rows, scales and row weights of tokens `toks`, bit for bit."""
    sub_dst = dst[toks]
    valid = sub_dst >= 0
    # oracle on the sampled tokens, written to compact rows 0..n-1
    compact = np.where(valid, np.arange(sub_dst.size).reshape(sub_dst.shape), -1).astype(np.int32)
    o_rows, o_sc, o_w = orc.dispatch(case["x"][toks], compact, sub_dst.size, w.quant,
                                     topk_w=case["w"][toks])
    sel = torch.from_numpy(sub_dst[valid].astype(np.int64)).to(g["out_rows"].device)
    osel = compact[valid]
    if w.quant == "none":
        got = to_np_u16(g["out_rows"].index_select(0, sel))
    else:
        got = g["out_rows"].index_select(0, sel).cpu().numpy()
    assert np.array_equal(got, o_rows[osel]), "dispatched rows differ from the oracle"
    if w.quant != "none":
        gs = g["out_scales"].index_select(0, sel).cpu().numpy()
        assert np.array_equal(gs.view(np.uint32), o_sc[osel].view(np.uint32)), "scales differ"
    if check_row_w:
        assert np.array_equal(g["row_w"].index_select(0, sel).cpu().numpy().view(np.uint32),
                              o_w[osel].view(np.uint32))


def check_combine(w, case, g, ref, sample_tokens=None, seed=0, orc=None):
    """GPU combine vs oracle on the same y bytes; returns the exact-match fraction."""
    orc = orc or oracle.default()
    T, K = case["idx"].shape
    if T == 0:
        return 1.0
    dst = ref["dst_row"]
    if sample_tokens is None or sample_tokens >= T:
        toks = np.arange(T)
    else:
        rng = np.random.default_rng(seed + 1)
        toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, sample_tokens, replace=False)]))
    exact = 0
    worst = 0
    for c0 in range(0, toks.size, CHUNK_TOKENS):
        part = toks[c0:c0 + CHUNK_TOKENS]
        sub = dst[part]
        flat = sub.ravel()
        gather = torch.from_numpy(np.where(flat >= 0, flat, 0).astype(np.int64)).to(g["y"].device)
        y_c = to_np_u16(g["y"].index_select(0, gather))
        compact = np.where(sub >= 0, np.arange(sub.size).reshape(sub.shape), -1).astype(np.int32)
        ref_out = orc.combine(y_c, case["w"][part], compact, w.H)
        got = to_np_u16(g["out"].index_select(0, torch.from_numpy(part).to(g["out"].device)))
        d = bf16_ulp_diff(got, ref_out)
        worst = max(worst, int(d.max()))
        exact += int((d == 0).sum())
    assert worst <= 1, f"combine differs by {worst} bf16 ulp"
    return exact / float(toks.size * w.H)


def check_dispatch_mn(w, case, L, out_rows, out_scales, ref, orc=None, sentinel=None):
    """MN-major UE8M0 dispatch: rows bit-exact on every valid row; scale words
    bit-exact against the oracle's re-layout of its row-major words."""
    orc = orc or oracle.default()
    cap_rows = L.rows_capacity
    o_rows, o_sc, _ = orc.dispatch(case["x"], ref["dst_row"], max(cap_rows, 1), "fp8_ue8m0")
    valid = np.nonzero(ref["row_src"] >= 0)[0]
    if valid.size == 0:
        return
    got_rows = out_rows[:ref["rows"]].cpu().numpy()
    assert np.array_equal(got_rows[valid], o_rows[valid]), "dispatched rows differ"
    mn = orc.scales_mn_major(o_sc[:cap_rows], w.layout, E=w.E, cap=w.cap)
    got = out_scales.reshape(-1).cpu().numpy()
    assert got.size == mn.size
    P = o_sc.shape[1]
    if w.layout == "masked":
        stride = (w.cap + 3) // 4 * 4
        pos = ((valid // w.cap)[:, None] * P + np.arange(P)[None, :]) * stride + \
            (valid % w.cap)[:, None]
    else:
        stride = (cap_rows + 3) // 4 * 4
        pos = np.arange(P)[None, :] * stride + valid[:, None]
    assert np.array_equal(got[pos.ravel()], mn[pos.ravel()]), "MN-major scale words differ"
