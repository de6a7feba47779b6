"""CPU oracle for MoE token dispatch / combine -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around the plain-C oracle in ``oracle.c``.  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import this
package; the library under ``combine_expert_histogram_gb300`` never does, and
the two share no code.  See ``oracle.h`` for what each function computes and
which choices are "parity unpinned".

``Oracle(path)`` wraps one compiled copy of the oracle (the tests also load
deliberately broken copies to show that the pins catch them); the module-level
functions use the default build, ``liboracle.so`` next to the source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, CAPACITY, BAD_EXPERT_ID = 0, 2, 3
QUANT = {"none": 0, "fp8_f32": 1, "fp8_ue8m0": 2, "mxfp8": 3}

GCC_FLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_oracle(src: str, out: str, include_dir: str = _HERE) -> str:
    """Compile one copy of the oracle source into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-I", include_dir, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its source."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(SRC), os.path.getmtime(HDR)))
    if force or stale:
        compile_oracle(SRC, _LIB)
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def rows_capacity(T, K, E, align, layout, cap=0):
    """Rows a row buffer must hold for this layout (contiguous: the worst case)."""
    if layout == "masked":
        return E * cap
    return T * K + min(E, T * K) * (align - 1)


def scale_cols(H: int, quant: str) -> int:
    """fp32 / int32 scale words per row."""
    G = H // 128
    if quant in ("fp8_f32", "mxfp8"):
        return G  # fp32 words, or 4 E8M0 bytes per int32 word
    return (G + 3) // 4 if quant == "fp8_ue8m0" else 0


class Oracle:
    """One loaded copy of the C oracle."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int
        L.orc_bf16_round.restype = ctypes.c_uint16
        L.orc_bf16_round.argtypes = [ctypes.c_float]
        L.orc_bf16_to_float.restype = ctypes.c_float
        L.orc_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_quant_group_f32.restype = None
        L.orc_quant_group_f32.argtypes = [P, I, P, P]
        L.orc_quant_group_ue8m0.restype = None
        L.orc_quant_group_ue8m0.argtypes = [P, I, P, P]
        L.orc_quant_block_mx.restype = None
        L.orc_quant_block_mx.argtypes = [P, I, P, P]
        L.orc_layout.restype = I
        L.orc_layout.argtypes = [P, I, I, I, I, I, I, I, P, P, P, P, P]
        L.orc_dispatch.restype = None
        L.orc_dispatch.argtypes = [P, I, I, I, I, P, P, P, P, P]
        L.orc_combine.restype = None
        L.orc_combine.argtypes = [P, P, P, I, I, I, P]
        L.orc_route_topk.restype = None
        L.orc_route_topk.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
        L.orc_rank_ids.restype = None
        L.orc_rank_ids.argtypes = [P, I, I, I, I, P]
        L.orc_rank_expand.restype = None
        L.orc_rank_expand.argtypes = [P, I, I, I, I, P, P, I, I, P, P, P, P]
        L.orc_scales_mn_major.restype = None
        L.orc_scales_mn_major.argtypes = [P, I, I, I, I, I, P]
        L.orc_masked_repack.restype = I
        L.orc_masked_repack.argtypes = [P, P, I, I, P, P, I, I, P, P, P]
        self.lib = L
        self.path = path

    # ------------------------------------------------------------- scalars
    def bf16_round(self, f: float) -> int:
        return int(self.lib.orc_bf16_round(float(f)))

    def bf16_round_array(self, a: np.ndarray) -> np.ndarray:
        f = self.lib.orc_bf16_round
        return np.array([f(float(v)) for v in np.asarray(a, dtype=np.float32).ravel()],
                        dtype=np.uint16)

    def bf16_to_float(self, b: int) -> float:
        return float(self.lib.orc_bf16_to_float(int(b)))

    def e4m3_encode(self, v: float) -> int:
        return int(self.lib.orc_e4m3_encode(float(v)))

    def e4m3_encode_array(self, a: np.ndarray) -> np.ndarray:
        f = self.lib.orc_e4m3_encode
        return np.array([f(float(v)) for v in np.asarray(a, dtype=np.float32).ravel()],
                        dtype=np.uint8)

    def e4m3_decode(self, c: int) -> float:
        return float(self.lib.orc_e4m3_decode(int(c)))

    def quant_group(self, x_bits: np.ndarray, mode: str):
        """Quantise one group: (q uint8 [n], fp32 scale | UE8M0 / E8M0 byte)."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        q = np.zeros(x.size, dtype=np.uint8)
        if mode == "fp8_f32":
            s = np.zeros(1, dtype=np.float32)
            self.lib.orc_quant_group_f32(_p(x), x.size, _p(q), _p(s))
            return q, float(s[0])
        e = np.zeros(1, dtype=np.uint8)
        if mode == "mxfp8":
            self.lib.orc_quant_block_mx(_p(x), x.size, _p(q), _p(e))
        else:
            self.lib.orc_quant_group_ue8m0(_p(x), x.size, _p(q), _p(e))
        return q, int(e[0])

    # --------------------------------------------------------------- layout
    def layout(self, topk_idx: np.ndarray, E: int, layout: str = "contig", align: int = 128,
               cap: int = 0, R: int = 1):
        """dict(count, offset, dst_row [T,K], row_src [rows], rank_rows, status, rows)."""
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        T, K = idx.shape
        masked = 1 if layout == "masked" else 0
        count = np.zeros(E, dtype=np.int32)
        offset = np.zeros(E + 1, dtype=np.int32)
        dst = np.zeros(T * K, dtype=np.int32)
        nrows = rows_capacity(T, K, E, align, layout, cap)
        row_src = np.full(max(nrows, 1), -7, dtype=np.int32)
        rank_rows = np.zeros(R, dtype=np.int32)
        st = self.lib.orc_layout(_p(idx), T, K, E, R, masked, align, cap, _p(count),
                                 _p(offset), _p(dst), _p(row_src), _p(rank_rows))
        rows = int(offset[E])
        return dict(count=count, offset=offset, dst_row=dst.reshape(T, K),
                    row_src=row_src[:rows], rank_rows=rank_rows, status=int(st), rows=rows)

    # ------------------------------------------------------------- dispatch
    def dispatch(self, x_bits: np.ndarray, dst_row: np.ndarray, rows: int, quant: str,
                 topk_w: np.ndarray | None = None, fill: int = 0):
        """(out_rows, out_scales, row_w); rows never written keep ``fill``."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        T, H = x.shape
        d = np.ascontiguousarray(dst_row, dtype=np.int32)
        K = d.shape[1] if d.ndim == 2 else (d.size // T if T else 0)
        if quant == "none":
            out = np.full((rows, H), fill, dtype=np.uint16)
            sc = None
        else:
            out = np.full((rows, H), fill, dtype=np.uint8)
            dt = np.float32 if quant == "fp8_f32" else np.int32  # mxfp8: 4 E8M0 bytes per word
            sc = np.zeros((rows, scale_cols(H, quant)), dtype=dt)
        row_w = w = None
        if topk_w is not None:
            w = np.ascontiguousarray(topk_w, dtype=np.float32)
            row_w = np.zeros(rows, dtype=np.float32)
        self.lib.orc_dispatch(_p(x), T, K, H, QUANT[quant], _p(d), _p(out), _p(sc), _p(w),
                              _p(row_w))
        return out, sc, row_w

    # -------------------------------------------------------------- combine
    def combine(self, y_bits: np.ndarray, topk_w: np.ndarray, dst_row: np.ndarray, H: int):
        """bf16 bits [T, H]; y_bits is [rows, H], dst_row / topk_w are [T, K]."""
        y = np.ascontiguousarray(y_bits, dtype=np.uint16)
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        d = np.ascontiguousarray(dst_row, dtype=np.int32)
        T, K = d.shape
        out = np.zeros((T, H), dtype=np.uint16)
        self.lib.orc_combine(_p(y), _p(w), _p(d), T, K, H, _p(out))
        return out

    # ------------------------------------------------------------ router top-k
    def route_topk(self, logits: np.ndarray, K: int, mode: str = "softmax",
                   bias: np.ndarray | None = None, n_group: int = 1, topk_group: int = 1):
        """(topk_idx int32 [T,K], topk_w float64 [T,K], selection score fp32 [T,K])."""
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = lg.shape
        idx = np.zeros((T, K), dtype=np.int32)
        w = np.zeros((T, K), dtype=np.float64)
        sc = np.zeros((T, K), dtype=np.float32)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        m = {"softmax": 0, "grouped_sigmoid": 1}[mode]
        self.lib.orc_route_topk(_p(lg), _p(b), T, E, K, m, n_group, topk_group, _p(idx),
                                _p(w), _p(sc))
        return idx, w, sc

    # ------------------------------------------ per-rank deduplicated sending
    def rank_ids(self, topk_idx: np.ndarray, E: int, R: int) -> np.ndarray:
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        T, K = idx.shape
        out = np.zeros((T, K), dtype=np.int32)
        self.lib.orc_rank_ids(_p(idx), T, K, E, R, _p(out))
        return out

    def rank_layout(self, topk_idx: np.ndarray, E: int, R: int, align: int = 1):
        """The rank-major send layout: orc_layout over first-occurrence rank ids."""
        return self.layout(self.rank_ids(topk_idx, E, R), R, "contig", align=align)

    def rank_expand(self, topk_idx, E, R, send_dst, dst_row, rows, send_rows, send_scales,
                    fill=0):
        """Expert-layout rows [rows, ...] filled from the send buffer."""
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        T, K = idx.shape
        sr = np.ascontiguousarray(send_rows)
        out = np.full((rows,) + sr.shape[1:], fill, dtype=sr.dtype)
        row_bytes = sr.shape[1] * sr.dtype.itemsize if sr.ndim > 1 else sr.dtype.itemsize
        ss = oscales = None
        scale_bytes = 0
        if send_scales is not None:
            ss = np.ascontiguousarray(send_scales)
            oscales = np.zeros((rows,) + ss.shape[1:], dtype=ss.dtype)
            scale_bytes = ss.shape[1] * ss.dtype.itemsize
        self.lib.orc_rank_expand(_p(idx), T, K, E, R,
                                 _p(np.ascontiguousarray(send_dst, dtype=np.int32)),
                                 _p(np.ascontiguousarray(dst_row, dtype=np.int32)),
                                 row_bytes, scale_bytes, _p(sr), _p(ss), _p(out), _p(oscales))
        return out, oscales

    # ------------------------------------------------- MN-major scale layout
    def scales_mn_major(self, row_major: np.ndarray, layout: str, E: int = 0, cap: int = 0,
                        fill: int = 0) -> np.ndarray:
        """Row-major packed UE8M0 words [rows, P] -> the MN-major buffer (1-D int32)."""
        rm = np.ascontiguousarray(row_major, dtype=np.int32)
        rows, P = rm.shape
        if layout == "masked":
            n = E * P * ((cap + 3) // 4 * 4)
        else:
            n = P * ((rows + 3) // 4 * 4)
        out = np.full(max(n, 1), fill, dtype=np.int32)[:n]
        self.lib.orc_scales_mn_major(_p(rm), rows, P, 1 if layout == "masked" else 0, E, cap,
                                     _p(out))
        return out

    # --------------------------------------------------------- masked repack
    def masked_repack(self, rows_buf: np.ndarray, scales, H: int, quant: str,
                      offset: np.ndarray, count: np.ndarray, E: int, cap: int, fill: int = 0):
        """(slab [E*cap, ...], slab_scales, masked_m, status)."""
        rb = np.ascontiguousarray(rows_buf)
        slab = np.full((E * cap,) + rb.shape[1:], fill, dtype=rb.dtype)
        sb = ss = None
        if scales is not None:
            sb = np.ascontiguousarray(scales)
            ss = np.zeros((E * cap,) + sb.shape[1:], dtype=sb.dtype)
        mm = np.zeros(E, dtype=np.int32)
        st = self.lib.orc_masked_repack(_p(rb), _p(sb), H, QUANT[quant],
                                        _p(np.ascontiguousarray(offset, dtype=np.int32)),
                                        _p(np.ascontiguousarray(count, dtype=np.int32)),
                                        E, cap, _p(slab), _p(ss), _p(mm))
        return slab, ss, mm, int(st)


_lock = threading.Lock()
_default = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def __getattr__(name):
    # module-level convenience: oracle.layout(...) == oracle.default().layout(...)
    if name in ("bf16_round", "bf16_round_array", "bf16_to_float", "e4m3_encode",
                "e4m3_encode_array", "e4m3_decode", "quant_group", "layout", "dispatch",
                "combine", "masked_repack", "scales_mn_major", "rank_ids", "rank_layout",
                "rank_expand", "route_topk"):
        return getattr(default(), name)
    raise AttributeError(name)
