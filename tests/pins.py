"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  The same pins run against the real oracle (they must pass) and
against deliberately broken copies of it (each copy must fail at least one).

What the pins compare with:
  * torch's CPU casts to bfloat16 and float8_e4m3fn (independent library code),
  * the format definitions' special points (tests/golden/*.txt, cited there),
  * brute force: nearest-code search with ties to even, O((TK)^2) slot counting,
  * exact rational arithmetic (fractions) for "correctly rounded" divides,
  * closed forms and invariants: counts sum to T*K, segments are aligned,
    dst_row is injective, combine(dispatch(x)) with identity experts.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ brute force
def _e4m3_table():
    codes = np.arange(0x00, 0x7F, dtype=np.uint8)  # all finite non-negative codes
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


_CODES, _VALS = _e4m3_table()


def e4m3_nearest(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code to each float64 value, ties to the even code.

    Saturation needs no special case: above 448 the nearest finite value is 448.
    """
    v = np.asarray(v, dtype=np.float64).ravel()
    a = np.minimum(np.abs(v), 512.0)  # keeps distances resolvable; order unchanged above 448
    d = np.abs(a[:, None] - _VALS[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    n = cand.sum(axis=1)
    assert (n >= 1).all() and (n <= 2).all()
    even = (_CODES % 2 == 0)[None, :]
    pick_even = cand & even
    choose = np.where((n == 2)[:, None], pick_even, cand)
    code = _CODES[np.argmax(choose, axis=1)]
    return (code | np.where(np.signbit(v), 0x80, 0x00)).astype(np.uint8)


def torch_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _f32(x) -> float:
    return float(np.float32(x))


def _read_points(name):
    pts = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                v, c = line.split()
                pts.append((float(v), int(c, 16)))
    return pts


# -------------------------------------------------------------------- bf16
def pin_bf16(orc, rng):
    bits = rng.integers(0, 2**32, size=4000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # exact halfway cases with both parities of the kept bit, and near-overflow
    hw = (rng.integers(0, 2**16, size=400, dtype=np.uint32) << 16) | 0x8000
    hw_f = hw.view(np.float32)
    hw_f = hw_f[np.isfinite(hw_f)]
    extra = np.array([0.0, -0.0, 1.0, -1.0, 3.3895e38, 3.4e38, -3.4e38, 1e-40, -1e-40,
                      1.00390625, 1.01171875], dtype=np.float32)
    allv = np.concatenate([f, hw_f, extra]).astype(np.float32)
    got = orc.bf16_round_array(allv)
    exp = torch_bf16_bits(allv)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"bf16 rounding differs from torch at {allv[bad[:5]]}"
    for v, bits_ in _read_points("bf16_spec_points.txt"):
        assert orc.bf16_round(v) == bits_, (v, hex(bits_))
        assert orc.bf16_to_float(bits_) == _f32(v)


# -------------------------------------------------------------------- E4M3
def pin_e4m3_decode(orc, rng):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


def pin_e4m3_roundtrip_and_ties(orc, rng):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = orc.e4m3_decode(c)
        assert orc.e4m3_encode(v) == c, hex(c)
    # midpoints between adjacent finite codes of one sign go to the even code
    for c in range(0x00, 0x7E):
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = (lo + hi) / 2.0  # <= 5 significant bits: exact in fp32
        assert _f32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == even, (hex(c), mid)
        assert orc.e4m3_encode(-mid) == even | 0x80, (hex(c), -mid)


def pin_e4m3_nearest(orc, rng):
    mag = np.exp2(rng.uniform(-13.0, 9.5, size=6000))
    sgn = np.where(rng.random(6000) < 0.5, -1.0, 1.0)
    v = (mag * sgn).astype(np.float32)
    v = np.concatenate([v, np.array([0.0, -0.0, -1e-30, 1e-30, 448.0, 449.0, 463.9, 464.0,
                                     1e6, -1e6, 3e38, -3e38], dtype=np.float32)])
    got = orc.e4m3_encode_array(v)
    exp = e4m3_nearest(v.astype(np.float64))
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"E4M3 encode differs from nearest-even at {v[bad[:5]]}"
    # torch's cast (round to nearest even) on the range where it does not overflow
    inr = v[np.abs(v) < 464.0]
    tc = torch.from_numpy(inr.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode_array(inr), tc)
    for val, code in _read_points("e4m3_spec_points.txt"):
        assert orc.e4m3_encode(val) == code, (val, hex(code))
        d = orc.e4m3_decode(code)
        assert d == val and math.copysign(1, d) == math.copysign(1, val)


# ------------------------------------------------------------------- quant
def _groups(rng, n=120):
    out = []
    for i in range(n):
        kind = i % 6
        if kind == 0:
            g = rng.standard_normal(128)
        elif kind == 1:
            g = rng.standard_normal(128) * 10.0 ** rng.uniform(-8, 8)
        elif kind == 2:
            g = np.zeros(128)
        elif kind == 3:
            g = rng.standard_normal(128) * 1e-6  # amax below the 1e-4 clamp
        elif kind == 4:
            g = rng.standard_normal(128) * 1e-3
            g[rng.integers(0, 128)] = 1e4  # one outlier
        else:
            g = np.round(rng.standard_normal(128) * 4) / 4  # many exact ties
        out.append(torch_bf16_bits(g.astype(np.float32)))
    return out


def _correctly_rounded_div(num: float, den: float) -> float:
    """IEEE binary32 quotient num/den rounded to nearest-even, by exact fractions."""
    exact = Fraction(num) / Fraction(den)
    q = np.float32(num) / np.float32(den)  # candidate; verified below, not trusted
    cands = [np.nextafter(q, np.float32(-np.inf)), q, np.nextafter(q, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - exact),
                                     int(np.float32(c).view(np.uint32)) & 1))
    return float(best)


def pin_quant_f32(orc, rng):
    for xb in _groups(rng):
        x = bf16_bits_to_f32(xb).astype(np.float64)
        q, s = orc.quant_group(xb, "fp8_f32")
        amax = float(np.abs(x).max())
        clamped = max(_f32(amax), _f32(1e-4))
        assert s == _correctly_rounded_div(clamped, 448.0), (amax, s)
        # the encode step against brute force on the fp32 quotients
        quot = np.array([_correctly_rounded_div(float(xi), s) if xi != 0 else 0.0 * xi
                         for xi in x])
        assert np.array_equal(q, e4m3_nearest(quot))
        dq = np.array([orc.e4m3_decode(int(c)) for c in q])
        if amax >= 1e-4:
            assert np.abs(dq).max() == 448.0
        # dequantisation error: half an E4M3 ulp of |x/s| (normal) or 2^-10 (subnormal)
        err = np.abs(x - dq * s)
        bound = np.where(np.abs(x / s) >= 2.0 ** -6, np.abs(x / s) * 2.0 ** -4, 2.0 ** -10) * s
        assert (err <= bound * (1 + 1e-6) + 1e-30).all()


def pin_quant_ue8m0(orc, rng):
    for xb in _groups(rng):
        x = bf16_bits_to_f32(xb).astype(np.float64)
        q, e = orc.quant_group(xb, "fp8_ue8m0")
        amax = float(np.abs(x).max())
        s = _correctly_rounded_div(max(_f32(amax), _f32(1e-4)), 448.0)
        # e is the smallest exponent with s <= 2^(e-127)
        assert math.ldexp(1.0, e - 128) < s <= math.ldexp(1.0, e - 127), (s, e)
        v = x * math.ldexp(1.0, 127 - e)  # exact in float64 and in fp32 here
        assert np.abs(v).max() <= 448.0  # rounding the scale up never saturates
        assert np.array_equal(q, e4m3_nearest(v))


def pin_quant_mx(orc, rng):
    """OCP MX conversion: X = 2^(floor(log2 amax) - 8), so amax / X lies in
    [256, 512) for every normal amax; E8M0 byte = log2 X + 127, clamped at 0."""
    blocks = [b[:32] for b in _groups(rng)] + [b[32:64] for b in _groups(rng, 24)]
    tiny = torch_bf16_bits(np.full(32, 2.0 ** -130, dtype=np.float32))  # subnormal block
    blocks.append(tiny)
    for xb in blocks:
        x = bf16_bits_to_f32(xb).astype(np.float64)
        q, byte = orc.quant_group(xb, "mxfp8")
        amax = float(np.abs(x).max())
        if amax >= 2.0 ** -126:
            _, ex = math.frexp(amax)  # amax = f * 2^ex, f in [0.5, 1)
            shared = ex - 1 - 8
            assert byte == max(0, shared + 127), (amax, byte)
            X = math.ldexp(1.0, byte - 127)
            if byte > 0:
                assert 256.0 <= amax / X < 512.0
        else:
            assert byte == 0  # zero and subnormal blocks: smallest E8M0 scale
        X = math.ldexp(1.0, byte - 127)
        assert np.array_equal(q, e4m3_nearest(x / X))  # saturates above 448


# ------------------------------------------------------------------ layout
def _check_layout(orc, idx, E, kind, align, cap, R):
    T, K = idx.shape
    L = orc.layout(idx, E, kind, align=align, cap=cap, R=R)
    flat = idx.ravel()
    valid = (flat >= 0) & (flat < E)
    cnt = np.bincount(flat[valid], minlength=E)
    assert np.array_equal(L["count"], cnt)
    assert L["count"].sum() == valid.sum()
    off = L["offset"]
    if kind == "contig":
        assert off[0] == 0
        seg = np.diff(off)
        assert (seg % align == 0).all() and (seg >= cnt).all() and (seg < cnt + align).all()
    else:
        assert np.array_equal(off, np.arange(E + 1) * cap)
    # brute-force slot: earlier entries (lexicographic (t,k) = flat order) with the same id
    exp_dst = np.full(T * K, -1, dtype=np.int64)
    overflow = False
    for i in range(T * K):
        e = flat[i]
        if not (0 <= e < E):
            continue
        slot = int(np.sum(flat[:i] == e))
        if kind == "masked" and slot >= cap:
            overflow = True
            continue
        exp_dst[i] = off[e] + slot
    assert np.array_equal(L["dst_row"].ravel(), exp_dst)
    bad = (~valid & (flat != -1)).any()
    exp_status = 3 if bad else (2 if overflow else 0)
    assert L["status"] == exp_status, (L["status"], exp_status)
    rows = L["rows"]
    assert rows == (E * cap if kind == "masked" else off[E])
    rs = L["row_src"]
    d = exp_dst[exp_dst >= 0]
    assert len(np.unique(d)) == d.size  # injective
    exp_rs = np.full(rows, -1, dtype=np.int64)
    exp_rs[d] = np.nonzero(exp_dst >= 0)[0]
    assert np.array_equal(rs, exp_rs)
    assert np.array_equal(L["rank_rows"], cnt.reshape(R, E // R).sum(axis=1))
    return L


def pin_layout_bruteforce(orc, rng):
    for it in range(250):
        T = int(rng.integers(0, 13))
        K = int(rng.integers(1, 5))
        E = int(rng.choice([1, 2, 3, 4, 6, 8]))
        R = int(rng.choice([r for r in (1, 2, 3, 4) if E % r == 0]))
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)  # repeats allowed
        if it % 3 == 0:
            idx = np.where(idx < 0, 0, idx).astype(np.int32)
        align = int(rng.choice([1, 2, 4, 8, 128]))
        _check_layout(orc, idx, E, "contig", align, 0, R)
        cap = int(rng.integers(1, max(2, T * K + 2)))
        _check_layout(orc, idx, E, "masked", 1, cap, R)


def pin_layout_bad_ids(orc, rng):
    idx = np.array([[0, 5], [-2, 1], [3, -1], [4, 4]], dtype=np.int32)
    L = _check_layout(orc, idx, 4, "contig", 4, 0, 2)
    assert L["status"] == 3
    assert L["dst_row"][0, 1] == -1 and L["dst_row"][1, 0] == -1 and L["dst_row"][2, 1] == -1


# ---------------------------------------------------------------- dispatch
def pin_dispatch(orc, rng):
    for quant, H in (("none", 256), ("fp8_f32", 384), ("fp8_ue8m0", 128), ("fp8_ue8m0", 384),
                     ("fp8_ue8m0", 7168), ("fp8_f32", 7168), ("mxfp8", 128), ("mxfp8", 640)):
        T, K, E = 9, 3, 5
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
        w = rng.random((T, K)).astype(np.float32)
        x = torch_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        L = orc.layout(idx, E, "contig", align=4)
        out, sc, roww = orc.dispatch(x, L["dst_row"], L["rows"], quant, topk_w=w,
                                     fill=0xAB if quant != "none" else 0xABCD)
        G = H // 128
        written = np.zeros(L["rows"], dtype=bool)
        for t in range(T):
            for k in range(K):
                r = L["dst_row"][t, k]
                if r < 0:
                    continue
                written[r] = True
                assert roww[r] == w[t, k]
                if quant == "none":
                    assert np.array_equal(out[r], x[t])
                    continue
                if quant == "mxfp8":
                    sb = sc[r].view(np.uint8)  # H/32 E8M0 bytes, 4 per int32 word
                    for b in range(H // 32):
                        q, byte = orc.quant_group(x[t, b * 32:(b + 1) * 32], quant)
                        assert np.array_equal(out[r, b * 32:(b + 1) * 32], q)
                        assert (int(sc[r, b // 4]) >> (8 * (b % 4))) & 0xFF == byte == sb[b]
                    continue
                for g in range(G):
                    q, s = orc.quant_group(x[t, g * 128:(g + 1) * 128], quant)
                    assert np.array_equal(out[r, g * 128:(g + 1) * 128], q)
                    if quant == "fp8_f32":
                        assert sc[r, g] == np.float32(s)
                    else:
                        word = int(sc[r, g // 4]) & 0xFFFFFFFF
                        assert (word >> (8 * (g % 4))) & 0xFF == s  # little-endian byte g%4
                if quant == "fp8_ue8m0":
                    for b in range(G, 4 * ((G + 3) // 4)):  # padding bytes hold 127 (2^0)
                        assert (int(sc[r, b // 4]) >> (8 * (b % 4))) & 0xFF == 127
        fill = 0xAB if quant != "none" else 0xABCD
        assert (out[~written] == fill).all()


# ----------------------------------------------------------------- combine
def pin_combine(orc, rng):
    T, H, E = 23, 256, 6
    x = torch_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xf = bf16_bits_to_f32(x).astype(np.float64)
    # (a) K = 1, w = 1: combine(dispatch(x)) is the inverse permutation -> exactly x
    idx1 = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    L = orc.layout(idx1, E, "contig", align=8)
    y, _, _ = orc.dispatch(x, L["dst_row"], L["rows"], "none")
    out = orc.combine(y, np.ones((T, 1), np.float32), L["dst_row"], H)
    assert np.array_equal(out, x)
    # (b) identity experts, K = 4, weights summing to 1: within 1 bf16 ulp of the
    #     exact sum (so never ~K*x: the reduction happens exactly once)
    K = 4
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    L = orc.layout(idx, E, "contig", align=8)
    y, _, _ = orc.dispatch(x, L["dst_row"], L["rows"], "none")
    out = bf16_bits_to_f32(orc.combine(y, w, L["dst_row"], H)).astype(np.float64)
    exact = (w.astype(np.float64).sum(axis=1))[:, None] * xf
    _within_bf16_ulp(out, exact, np.abs(exact))
    # (c) general expert outputs and -1 entries, against the fp64 sum
    idx[rng.random((T, K)) < 0.25] = -1
    L = orc.layout(idx, E, "contig", align=8)
    yb = torch_bf16_bits(rng.standard_normal((max(L["rows"], 1), H)).astype(np.float32))
    yf = bf16_bits_to_f32(yb).astype(np.float64)
    out = bf16_bits_to_f32(orc.combine(yb, w, L["dst_row"], H)).astype(np.float64)
    exact = np.zeros((T, H))
    mag = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            r = L["dst_row"][t, k]
            if r >= 0:
                exact[t] += float(w[t, k]) * yf[r]
                mag[t] += abs(float(w[t, k])) * np.abs(yf[r])
    _within_bf16_ulp(out, exact, mag)
    none = (L["dst_row"] < 0).all(axis=1)
    if none.any():
        assert (out[none] == 0).all()
    # (d) each product and each sum rounded to fp32 on its own (no fused
    #     multiply-add): w = 1 + 2^-20 on +(1 + 2^-5) and -(1 + 2^-5) gives two
    #     products whose fp32 rounding drops the same 2^-25, so they cancel to
    #     exactly +0; a fused multiply-add would keep -2^-25 (a bf16 value)
    y2 = torch_bf16_bits(np.array([[1 + 2.0 ** -5], [-(1 + 2.0 ** -5)]], dtype=np.float32))
    w2 = np.full((1, 2), 1 + 2.0 ** -20, dtype=np.float32)
    out2 = orc.combine(y2, w2, np.array([[0, 1]], dtype=np.int32), 1)
    assert int(out2[0, 0]) == 0x0000


def _within_bf16_ulp(out, exact, mag):
    """|out - exact| <= 1 bf16 ulp of |exact| (+ fp32 accumulation slack)."""
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    slack = 8 * 2.0 ** -24 * mag
    assert (np.abs(out - exact) <= ulp + slack + 1e-30).all()


# ------------------------------------------------------------------ repack
def pin_masked_repack(orc, rng):
    T, K, E, H = 20, 3, 5, 384
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = torch_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    for quant in ("none", "fp8_f32", "fp8_ue8m0", "mxfp8"):
        for cap in (T, 7):
            Lc = orc.layout(idx, E, "contig", align=16)
            Lm = orc.layout(idx, E, "masked", cap=cap)
            rows_c, sc_c, _ = orc.dispatch(x, Lc["dst_row"], Lc["rows"], quant)
            rows_m, sc_m, _ = orc.dispatch(x, Lm["dst_row"], Lm["rows"], quant)
            slab, ss, mm, st = orc.masked_repack(rows_c, sc_c, H, quant, Lc["offset"],
                                                 Lc["count"], E, cap)
            assert np.array_equal(mm, np.minimum(Lc["count"], cap))
            assert st == (2 if (Lc["count"] > cap).any() else 0)
            for e in range(E):
                for s in range(mm[e]):
                    assert np.array_equal(slab[e * cap + s], rows_m[e * cap + s])
                    if ss is not None:
                        assert np.array_equal(ss[e * cap + s], sc_m[e * cap + s])


def pin_fp8_roundtrip(orc, rng):
    """combine(dequant(dispatch_fp8(x))) with identity experts ~ sum_k w_k x (2^-4 rel;
    2^-3 for MXFP8, whose scale rule saturates the top of the block's binade)."""
    T, K, E, H = 12, 3, 4, 256
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    x = torch_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xf = bf16_bits_to_f32(x).astype(np.float64)
    L = orc.layout(idx, E, "contig", align=4)
    for quant in ("fp8_f32", "fp8_ue8m0", "mxfp8"):
        q, sc, _ = orc.dispatch(x, L["dst_row"], L["rows"], quant)
        dec = np.array([orc.e4m3_decode(c) for c in range(256)])[q]
        G = H // 128
        if quant == "fp8_f32":
            s = np.repeat(sc.astype(np.float64), 128, axis=1)
        elif quant == "mxfp8":
            eb = sc.view(np.uint8).reshape(sc.shape[0], -1).astype(np.float64)
            s = np.repeat(np.exp2(eb - 127), 32, axis=1)
        else:
            eb = sc.view(np.uint8).reshape(sc.shape[0], -1)[:, :G].astype(np.float64)
            s = np.repeat(np.exp2(eb - 127), 128, axis=1)
        y = torch_bf16_bits((dec * s).astype(np.float32))
        out = bf16_bits_to_f32(orc.combine(y, w, L["dst_row"], H)).astype(np.float64)
        exact = w.astype(np.float64).sum(axis=1)[:, None] * xf
        amax = np.abs(xf).max()
        # E4M3 rounding is within 2^-4 relative; the MX rule's scale puts the
        # block maximum in [256, 512) and clamps above 448: up to 2^-3 there
        rel = 2.0 ** -3 if quant == "mxfp8" else 2.0 ** -4
        assert (np.abs(out - exact) <= rel * np.abs(exact) + 2.0 ** -6 * amax).all()


def pin_scales_mn_major(orc, rng):
    """MN-major re-layout == numpy's transpose of the row-major words; every
    scale column starts on a 16-byte boundary."""
    for rows, P in ((13, 3), (16, 14), (1, 1), (130, 2)):
        rm = rng.integers(-2**31, 2**31 - 1, size=(rows, P), dtype=np.int64).astype(np.int32)
        out = orc.scales_mn_major(rm, "contig", fill=-7)
        rows4 = (rows + 3) // 4 * 4
        assert out.size == P * rows4 and (rows4 * 4) % 16 == 0
        grid = out.reshape(P, rows4)
        assert np.array_equal(grid[:, :rows].T, rm)
        assert (grid[:, rows:] == -7).all()
    for E, cap, P in ((3, 5, 2), (4, 8, 14), (2, 1, 1)):
        rm = rng.integers(-2**31, 2**31 - 1, size=(E * cap, P), dtype=np.int64).astype(np.int32)
        out = orc.scales_mn_major(rm, "masked", E=E, cap=cap, fill=-7)
        cap4 = (cap + 3) // 4 * 4
        grid = out.reshape(E, P, cap4)
        assert np.array_equal(grid[:, :, :cap].transpose(0, 2, 1).reshape(E * cap, P), rm)
        assert (grid[:, :, cap:] == -7).all()


def pin_rank_dedup(orc, rng):
    """Send layout by brute force (token t is sent to rank r iff one of its
    experts lies in r; ascending tokens inside each rank, ranks in order), and
    expand(dispatch into the send layout) == dispatch into the expert layout."""
    for it in range(60):
        T = int(rng.integers(0, 15))
        R = int(rng.choice([1, 2, 4]))
        E = R * int(rng.integers(1, 4))
        K = int(rng.integers(1, 5))
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
        RL = orc.rank_layout(idx, E, R, align=1)
        ranks = [set() if T else set() for _ in range(T)]
        for t in range(T):
            ranks[t] = {int(e) * R // E for e in idx[t] if e >= 0}
        counts = [sum(1 for t in range(T) if r in ranks[t]) for r in range(R)]
        assert list(RL["count"]) == counts
        expect_row = {}
        row = 0
        for r in range(R):
            for t in range(T):
                if r in ranks[t]:
                    expect_row[(t, r)] = row
                    row += 1
        assert RL["rows"] == row
        for t in range(T):
            seen = set()
            for k in range(K):
                e = idx[t, k]
                d = RL["dst_row"][t, k]
                if e < 0 or (e * R // E) in seen:
                    assert d == -1
                else:
                    seen.add(e * R // E)
                    assert d == expect_row[(t, e * R // E)]
        # composition: expand(send) == direct dispatch, for every quantisation
        H = 256
        x = torch_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        L = orc.layout(idx, E, "contig", align=4)
        for quant in ("none", "fp8_ue8m0", "mxfp8"):
            srows, ssc, _ = orc.dispatch(x, RL["dst_row"], RL["rows"], quant)
            drows, dsc, _ = orc.dispatch(x, L["dst_row"], L["rows"], quant, fill=3)
            erows, esc = orc.rank_expand(idx, E, R, RL["dst_row"], L["dst_row"], L["rows"],
                                         srows, ssc, fill=3)
            assert np.array_equal(erows, drows)
            if dsc is not None:
                assert np.array_equal(esc, dsc)


def pin_route_topk(orc, rng):
    """Router top-k against numpy/scipy restatements: stable argsort of the logits
    (softmax is monotone), scipy's softmax / expit for the weights, and the grouped
    selection written out with numpy in fp32; exact ties go to the lower id."""
    import scipy.special as sp
    for T, E, K in ((64, 8, 2), (40, 32, 5), (20, 16, 16)):
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[:T // 2] = np.round(lg[:T // 2], 1)  # many exact ties
        idx, w, _ = orc.route_topk(lg, K, "softmax")
        exp_idx = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :K]
        assert np.array_equal(idx, exp_idx)
        p = sp.softmax(lg.astype(np.float64), axis=1)
        sel = np.take_along_axis(p, exp_idx, axis=1)
        assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
    for T, E, K, G, TG in ((50, 32, 4, 4, 2), (30, 64, 8, 8, 4), (10, 16, 3, 2, 1)):
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[::3, :] = np.round(lg[::3, :])  # exact ties within groups
        bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
        idx, w, _ = orc.route_topk(lg, K, "grouped_sigmoid", bias=bias, n_group=G, topk_group=TG)
        s32 = (np.float32(1.0) / (np.float32(1.0) + np.exp(-lg))).astype(np.float32)
        c = (s32 + bias).astype(np.float32)
        gs = E // G
        top2 = -np.sort(-c.reshape(T, G, gs), axis=2)[:, :, :2]
        gscore = (top2[:, :, 0] + top2[:, :, 1]).astype(np.float32)
        keep_g = np.argsort(-gscore.astype(np.float64), axis=1, kind="stable")[:, :TG]
        mask = np.zeros((T, G), dtype=bool)
        np.put_along_axis(mask, keep_g, True, axis=1)
        cm = np.where(np.repeat(mask, gs, axis=1), c.astype(np.float64), -np.inf)
        exp_idx = np.argsort(-cm, axis=1, kind="stable")[:, :K]
        assert np.array_equal(idx, exp_idx)
        assert np.isin(idx // gs, keep_g).all()  # every pick lies in a kept group
        sg = sp.expit(lg.astype(np.float64))
        sel = np.take_along_axis(sg, exp_idx, axis=1)
        assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)


ALL_PINS = [pin_bf16, pin_e4m3_decode, pin_e4m3_roundtrip_and_ties, pin_e4m3_nearest,
            pin_quant_f32, pin_quant_ue8m0, pin_quant_mx, pin_layout_bruteforce, pin_layout_bad_ids,
            pin_dispatch, pin_combine, pin_masked_repack, pin_fp8_roundtrip,
            pin_scales_mn_major, pin_rank_dedup, pin_route_topk]
