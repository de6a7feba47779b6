"""Thin ctypes binding over the C ABI in include/ep.h (argument marshalling only).

Every step of the path runs in libep.so's CUDA kernels; this module only
allocates torch tensors for outputs the caller did not pass, fills the
``ep_layout_t`` struct and forwards raw pointers plus torch's current CUDA
stream.  There is no CPU fallback: if libep.so is missing or a tensor is not on
a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep.so")

(EP_OK, EP_ERR_INVALID_ARG, EP_ERR_CAPACITY, EP_ERR_BAD_EXPERT_ID, EP_ERR_CUDA, EP_ERR_UNSUPPORTED,
 EP_ERR_TIMEOUT) = range(7)
LAYOUT_KIND = {"contig": 0, "masked": 1}
QUANT = {"none": 0, "fp8_f32": 1, "fp8_ue8m0": 2, "mxfp8": 3, "fp8_ue8m0_mn": 4}
MAX_TOPK, MAX_EXPERTS, MAX_ALIGN = 32, 1024, 128


class EPError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_str(code)}" if what else status_str(code))


class _Layout(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_topk", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("num_ranks", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("align", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32),
        ("dst_row", ctypes.c_void_p),
        ("row_src", ctypes.c_void_p),
        ("expert_count", ctypes.c_void_p),
        ("expert_offset", ctypes.c_void_p),
        ("rank_rows", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


_lib = None

EXPORTS = ("ep_status_str", "ep_rows_capacity", "ep_scale_cols", "ep_scale_words",
           "ep_layout_workspace_bytes",
           "ep_layout", "ep_dispatch", "ep_layout_dispatch", "ep_combine", "ep_masked_repack",
           "ep_layout_noalloc", "ep_selftest_bounded_wait", "ep_selftest_cluster_wait",
           "ep_rank_layout", "ep_rank_expand", "ep_route_topk")
NOALLOC_SCRATCH_BYTES = 256 * 1024


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libep.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    LP = ctypes.POINTER(_Layout)
    L.ep_status_str.restype = ctypes.c_char_p
    L.ep_status_str.argtypes = [ctypes.c_int]
    L.ep_rows_capacity.restype = I64
    L.ep_rows_capacity.argtypes = [LP]
    L.ep_scale_cols.restype = I64
    L.ep_scale_cols.argtypes = [I32, ctypes.c_int]
    L.ep_scale_words.restype = I64
    L.ep_scale_words.argtypes = [LP, I32, ctypes.c_int]
    L.ep_layout_workspace_bytes.restype = SZ
    L.ep_layout_workspace_bytes.argtypes = [LP]
    L.ep_layout.restype = ctypes.c_int
    L.ep_layout.argtypes = [P, LP, P, SZ, P]
    L.ep_dispatch.restype = ctypes.c_int
    L.ep_dispatch.argtypes = [LP, P, I32, ctypes.c_int, P, P, P, P, P]
    L.ep_layout_dispatch.restype = ctypes.c_int
    L.ep_layout_dispatch.argtypes = [P, LP, P, SZ, P, I32, ctypes.c_int, P, P, P, P, P]
    L.ep_combine.restype = ctypes.c_int
    L.ep_combine.argtypes = [LP, P, I32, P, P, P]
    L.ep_masked_repack.restype = ctypes.c_int
    L.ep_masked_repack.argtypes = [LP, P, P, I32, ctypes.c_int, I32, P, P, P, P]
    L.ep_route_topk.restype = ctypes.c_int
    L.ep_route_topk.argtypes = [P, P, I32, I32, I32, ctypes.c_int, I32, I32, P, P, P]
    L.ep_rank_layout.restype = ctypes.c_int
    L.ep_rank_layout.argtypes = [P, I32, P, LP, P, SZ, P]
    L.ep_rank_expand.restype = ctypes.c_int
    L.ep_rank_expand.argtypes = [LP, LP, P, I32, ctypes.c_int, P, P, P, P, P]
    L.ep_selftest_bounded_wait.restype = ctypes.c_int
    L.ep_selftest_bounded_wait.argtypes = [P, I64, P]
    L.ep_selftest_cluster_wait.restype = ctypes.c_int
    L.ep_selftest_cluster_wait.argtypes = [P, I64, P]
    L.ep_layout_noalloc.restype = ctypes.c_int
    L.ep_layout_noalloc.argtypes = [P, LP, P]
    if path == LIB_PATH:
        _lib = L
    return L


def status_str(code: int) -> str:
    try:
        return load_library().ep_status_str(int(code)).decode()
    except RuntimeError:
        return f"ep_status_t {code}"


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libep works on CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libep needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, what: str):
    if code != EP_OK:
        raise EPError(code, what)


@dataclass
class Layout:
    """Shape + device arrays of one layout (the dispatch "handle")."""

    num_tokens: int
    num_topk: int
    num_experts: int
    num_ranks: int
    kind: str
    align: int
    capacity: int
    max_tokens: int
    dst_row: torch.Tensor
    row_src: Optional[torch.Tensor]
    expert_count: torch.Tensor
    expert_offset: torch.Tensor
    rank_rows: Optional[torch.Tensor]
    status: torch.Tensor
    workspace: Optional[torch.Tensor] = None
    _c: _Layout = field(default=None, repr=False)

    def struct(self) -> _Layout:
        c = _Layout()
        c.num_tokens, c.num_topk, c.num_experts = self.num_tokens, self.num_topk, self.num_experts
        c.num_ranks, c.kind, c.align = self.num_ranks, LAYOUT_KIND[self.kind], self.align
        c.capacity, c.max_tokens = self.capacity, self.max_tokens
        c.dst_row = _ptr(self.dst_row).value
        c.row_src = _ptr(self.row_src).value if self.row_src is not None else None
        c.expert_count = _ptr(self.expert_count).value
        c.expert_offset = _ptr(self.expert_offset).value
        c.rank_rows = _ptr(self.rank_rows).value if self.rank_rows is not None else None
        c.status = _ptr(self.status).value
        self._c = c
        return c

    @property
    def rows_capacity(self) -> int:
        return ep_rows_capacity(self)

    def check_status(self) -> None:
        """Synchronise and raise EPError if a device-side error was recorded."""
        st = int(self.status.item())
        if st != EP_OK:
            raise EPError(st, "device status")


def new_layout(num_tokens: int, num_topk: int, num_experts: int, kind: str = "contig",
               align: int = 128, capacity: int = 0, num_ranks: int = 1, max_tokens: int = 0,
               with_row_src: bool = True, device=None) -> Layout:
    """Allocate the arrays of a layout (uninitialised; ep_layout fills them)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    i32 = dict(dtype=torch.int32, device=dev)
    L = Layout(num_tokens, num_topk, num_experts, num_ranks, kind, align, capacity, max_tokens,
               dst_row=torch.empty(max(num_tokens * num_topk, 1), **i32),
               row_src=None, expert_count=torch.empty(num_experts, **i32),
               expert_offset=torch.empty(num_experts + 1, **i32),
               rank_rows=torch.empty(num_ranks, **i32), status=torch.zeros(1, **i32))
    rows = ep_rows_capacity(L)
    if rows < 0:
        raise EPError(EP_ERR_INVALID_ARG, "layout shape")
    if with_row_src:
        L.row_src = torch.empty(max(rows, 1), **i32)
    ws = ep_layout_workspace_bytes(L)
    if ws:
        L.workspace = torch.empty((ws + 3) // 4, **i32)
    return L


# ------------------------------------------------------------- C ABI mirrors
def ep_rows_capacity(layout: Layout) -> int:
    c = _Layout()
    c.num_tokens, c.num_topk, c.num_experts = layout.num_tokens, layout.num_topk, layout.num_experts
    c.num_ranks, c.kind, c.align = layout.num_ranks, LAYOUT_KIND[layout.kind], layout.align
    c.capacity, c.max_tokens = layout.capacity, layout.max_tokens
    return int(load_library().ep_rows_capacity(ctypes.byref(c)))


def ep_scale_cols(hidden: int, quant: str) -> int:
    return int(load_library().ep_scale_cols(hidden, QUANT[quant]))


def _shape_struct(layout: Layout) -> _Layout:
    c = _Layout()
    c.num_tokens, c.num_topk, c.num_experts = layout.num_tokens, layout.num_topk, layout.num_experts
    c.num_ranks, c.kind, c.align = layout.num_ranks, LAYOUT_KIND[layout.kind], layout.align
    c.capacity, c.max_tokens = layout.capacity, layout.max_tokens
    return c


def ep_scale_words(layout: Layout, hidden: int, quant: str) -> int:
    return int(load_library().ep_scale_words(ctypes.byref(_shape_struct(layout)), hidden,
                                             QUANT[quant]))


def scale_buffer(layout: Layout, hidden: int, quant: str, device=None) -> Optional[torch.Tensor]:
    """An uninitialised scale buffer shaped for ``quant`` on this layout."""
    if quant == "none":
        return None
    dev = device if device is not None else layout.dst_row.device
    cols = ep_scale_cols(hidden, quant)
    if quant == "fp8_ue8m0_mn":
        if layout.kind == "masked":
            shape = (layout.num_experts, cols, (layout.capacity + 3) // 4 * 4)
        else:
            shape = (cols, (max(layout.rows_capacity, 1) + 3) // 4 * 4)
        return torch.empty(shape, device=dev, dtype=torch.int32)
    return torch.empty((max(layout.rows_capacity, 1), cols), device=dev,
                       dtype=torch.float32 if quant == "fp8_f32" else torch.int32)


def ep_layout_workspace_bytes(layout: Layout) -> int:
    c = _Layout()
    c.num_tokens, c.num_topk, c.num_experts = layout.num_tokens, layout.num_topk, layout.num_experts
    c.num_ranks, c.kind, c.align = layout.num_ranks, LAYOUT_KIND[layout.kind], layout.align
    c.capacity, c.max_tokens = layout.capacity, layout.max_tokens
    return int(load_library().ep_layout_workspace_bytes(ctypes.byref(c)))


def ep_layout(topk_idx: torch.Tensor, num_experts: int, kind: str = "contig", align: int = 128,
              capacity: int = 0, num_ranks: int = 1, max_tokens: int = 0,
              with_row_src: bool = True, out: Optional[Layout] = None, stream=None) -> Layout:
    """Expert histogram, padded scan and stable slots for topk_idx (int32 [T, K])."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise ValueError("topk_idx must be int32 [T, K]")
    T, K = topk_idx.shape
    L = out if out is not None else new_layout(T, K, num_experts, kind, align, capacity,
                                               num_ranks, max_tokens, with_row_src,
                                               device=topk_idx.device)
    if (L.num_tokens, L.num_topk) != (T, K):
        raise ValueError("layout shape does not match topk_idx")
    ws = L.workspace
    nbytes = ws.numel() * 4 if ws is not None else 0
    code = load_library().ep_layout(_ptr(topk_idx) if T * K else None, ctypes.byref(L.struct()),
                                    _ptr(ws), nbytes, _stream(stream))
    _check(code, "ep_layout")
    return L


def ep_dispatch(layout: Layout, x: torch.Tensor, quant: str = "none",
                out_rows: Optional[torch.Tensor] = None, out_scales: Optional[torch.Tensor] = None,
                topk_w: Optional[torch.Tensor] = None, row_w: Optional[torch.Tensor] = None,
                stream=None):
    """Scatter (and quantise) x (bf16 [T, H]) into the layout's rows.

    Returns (out_rows, out_scales, row_w).  out_rows is bf16 [rows, H] or uint8
    E4M3 bytes; out_scales fp32 [rows, H/128] (fp8_f32), int32 [rows, ceil(H/512)]
    (fp8_ue8m0) or int32 [rows, H/128] holding H/32 E8M0 bytes (mxfp8).
    """
    T, H = x.shape
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bf16")
    rows = layout.rows_capacity
    dev = x.device
    if out_rows is None:
        out_rows = torch.empty((max(rows, 1), H), device=dev,
                               dtype=torch.bfloat16 if quant == "none" else torch.uint8)
    if quant != "none" and out_scales is None:
        out_scales = scale_buffer(layout, H, quant, device=dev)
    if topk_w is not None and row_w is None:
        row_w = torch.empty(max(rows, 1), device=dev, dtype=torch.float32)
    code = load_library().ep_dispatch(ctypes.byref(layout.struct()), _ptr(x), H, QUANT[quant],
                                      _ptr(out_rows), _ptr(out_scales), _ptr(topk_w), _ptr(row_w),
                                      _stream(stream))
    _check(code, "ep_dispatch")
    return out_rows, out_scales, row_w


def ep_layout_dispatch(topk_idx: torch.Tensor, layout: Layout, x: torch.Tensor,
                       quant: str = "none", out_rows: Optional[torch.Tensor] = None,
                       out_scales: Optional[torch.Tensor] = None,
                       topk_w: Optional[torch.Tensor] = None, row_w: Optional[torch.Tensor] = None,
                       stream=None):
    """ep_layout into ``layout`` and ep_dispatch of x, in one call (the two
    kernels back to back).  Returns (out_rows, out_scales, row_w) like ep_dispatch."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise ValueError("topk_idx must be int32 [T, K]")
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bf16")
    T, K = topk_idx.shape
    if (layout.num_tokens, layout.num_topk) != (T, K):
        raise ValueError("layout shape does not match topk_idx")
    H = x.shape[1]
    rows = layout.rows_capacity
    dev = x.device
    if out_rows is None:
        out_rows = torch.empty((max(rows, 1), H), device=dev,
                               dtype=torch.bfloat16 if quant == "none" else torch.uint8)
    if quant != "none" and out_scales is None:
        out_scales = scale_buffer(layout, H, quant, device=dev)
    if topk_w is not None and row_w is None:
        row_w = torch.empty(max(rows, 1), device=dev, dtype=torch.float32)
    ws = layout.workspace
    code = load_library().ep_layout_dispatch(
        _ptr(topk_idx) if T * K else None, ctypes.byref(layout.struct()), _ptr(ws),
        ws.numel() * 4 if ws is not None else 0, _ptr(x), H, QUANT[quant], _ptr(out_rows),
        _ptr(out_scales), _ptr(topk_w), _ptr(row_w), _stream(stream))
    _check(code, "ep_layout_dispatch")
    return out_rows, out_scales, row_w


def ep_combine(layout: Layout, y: torch.Tensor, topk_w: torch.Tensor,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[t] = bf16(sum_k topk_w[t,k] * y[dst_row[t,k]]), fp32 accumulation."""
    H = y.shape[-1]
    if y.dtype != torch.bfloat16 or topk_w.dtype != torch.float32:
        raise ValueError("y must be bf16 and topk_w fp32")
    if out is None:
        out = torch.empty((layout.num_tokens, H), device=y.device, dtype=torch.bfloat16)
    code = load_library().ep_combine(ctypes.byref(layout.struct()), _ptr(y), H, _ptr(topk_w),
                                     _ptr(out), _stream(stream))
    _check(code, "ep_combine")
    return out


def ep_masked_repack(layout: Layout, rows: torch.Tensor, row_scales: Optional[torch.Tensor],
                     quant: str, capacity: int, slab: Optional[torch.Tensor] = None,
                     slab_scales: Optional[torch.Tensor] = None,
                     masked_m: Optional[torch.Tensor] = None, stream=None):
    """Contiguous layout rows -> masked slab [E, capacity, ...]; returns (slab, slab_scales, masked_m)."""
    E = layout.num_experts
    H = rows.shape[-1]
    dev = rows.device
    if slab is None:
        slab = torch.empty((E, capacity, H), device=dev, dtype=rows.dtype)
    if row_scales is not None and slab_scales is None:
        if quant == "fp8_ue8m0_mn":
            slab_scales = torch.empty((E, ep_scale_cols(H, quant), (capacity + 3) // 4 * 4),
                                      device=dev, dtype=row_scales.dtype)
        else:
            slab_scales = torch.empty((E, capacity, row_scales.shape[-1]), device=dev,
                                      dtype=row_scales.dtype)
    if masked_m is None:
        masked_m = torch.empty(E, device=dev, dtype=torch.int32)
    code = load_library().ep_masked_repack(ctypes.byref(layout.struct()), _ptr(rows),
                                           _ptr(row_scales), H, QUANT[quant], capacity, _ptr(slab),
                                           _ptr(slab_scales), _ptr(masked_m), _stream(stream))
    _check(code, "ep_masked_repack")
    return slab, slab_scales, masked_m


def ep_selftest_bounded_wait(status: torch.Tensor, limit_clocks: int, stream=None) -> None:
    """Make one bounded device wait run out; EP_ERR_TIMEOUT lands in ``status``."""
    if status.dtype != torch.int32 or not status.is_cuda:
        raise ValueError("status must be a device int32 tensor")
    _check(load_library().ep_selftest_bounded_wait(_ptr(status), int(limit_clocks),
                                                    _stream(stream)), "ep_selftest_bounded_wait")


def ep_selftest_cluster_wait(status: torch.Tensor, limit_clocks: int, stream=None) -> None:
    """Make the cluster exchange's bounded wait run out in a 2-CTA cluster;
    EP_ERR_TIMEOUT lands in ``status``."""
    if status.dtype != torch.int32 or not status.is_cuda:
        raise ValueError("status must be a device int32 tensor")
    _check(load_library().ep_selftest_cluster_wait(_ptr(status), int(limit_clocks),
                                                    _stream(stream)), "ep_selftest_cluster_wait")


def ep_layout_noalloc(topk_idx: torch.Tensor, out: Layout, stream=None) -> Layout:
    """ep_layout with the library's fixed scratch array instead of a workspace.

    For callers that cannot allocate device memory; ``out`` must be a layout
    whose arrays the caller already owns (``out.workspace`` is ignored).  Calls
    share the library's one scratch array, so calls that overlap on the GPU race.
    """
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise ValueError("topk_idx must be int32 [T, K]")
    T, K = topk_idx.shape
    if (out.num_tokens, out.num_topk) != (T, K):
        raise ValueError("layout shape does not match topk_idx")
    code = load_library().ep_layout_noalloc(_ptr(topk_idx) if T * K else None,
                                            ctypes.byref(out.struct()), _stream(stream))
    _check(code, "ep_layout_noalloc")
    return out


def ep_rank_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, align: int = 1,
                   out: Optional[Layout] = None, rank_idx: Optional[torch.Tensor] = None,
                   stream=None):
    """Per-rank deduplicated send layout; returns (rank Layout, rank_idx [T, K])."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise ValueError("topk_idx must be int32 [T, K]")
    T, K = topk_idx.shape
    RL = out if out is not None else new_layout(T, K, num_ranks, "contig", align=align,
                                                device=topk_idx.device)
    if rank_idx is None:
        rank_idx = torch.empty((T, K), dtype=torch.int32, device=topk_idx.device)
    ws = RL.workspace
    code = load_library().ep_rank_layout(_ptr(topk_idx) if T * K else None, num_experts,
                                         _ptr(rank_idx) if T * K else None,
                                         ctypes.byref(RL.struct()), _ptr(ws),
                                         ws.numel() * 4 if ws is not None else 0, _stream(stream))
    _check(code, "ep_rank_layout")
    return RL, rank_idx


def ep_rank_expand(rank_layout: Layout, layout: Layout, topk_idx: torch.Tensor, quant: str,
                   send_rows: torch.Tensor, send_scales: Optional[torch.Tensor],
                   out_rows: Optional[torch.Tensor] = None,
                   out_scales: Optional[torch.Tensor] = None, stream=None):
    """Send buffer -> per-expert rows (and scale rows); returns (out_rows, out_scales)."""
    H = send_rows.shape[-1]
    dev = send_rows.device
    rows = layout.rows_capacity
    if out_rows is None:
        out_rows = torch.empty((max(rows, 1), H), device=dev, dtype=send_rows.dtype)
    if send_scales is not None and out_scales is None:
        out_scales = torch.empty((max(rows, 1), send_scales.shape[-1]), device=dev,
                                 dtype=send_scales.dtype)
    code = load_library().ep_rank_expand(ctypes.byref(rank_layout.struct()),
                                         ctypes.byref(layout.struct()), _ptr(topk_idx), H,
                                         QUANT[quant], _ptr(send_rows), _ptr(send_scales),
                                         _ptr(out_rows), _ptr(out_scales), _stream(stream))
    _check(code, "ep_rank_expand")
    return out_rows, out_scales


ROUTE = {"softmax": 0, "grouped_sigmoid": 1}


def ep_route_topk(logits: torch.Tensor, num_topk: int, mode: str = "softmax",
                  bias: Optional[torch.Tensor] = None, n_group: int = 1, topk_group: int = 1,
                  topk_idx: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
                  stream=None):
    """Router top-k from fp32 logits [T, E]; returns (topk_idx int32, topk_w fp32) [T, K]."""
    if logits.dtype != torch.float32 or logits.dim() != 2:
        raise ValueError("logits must be fp32 [T, E]")
    T, E = logits.shape
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty((T, num_topk), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, num_topk), dtype=torch.float32, device=dev)
    code = load_library().ep_route_topk(_ptr(logits), _ptr(bias), T, E, num_topk, ROUTE[mode],
                                        n_group, topk_group, _ptr(topk_idx), _ptr(topk_w),
                                        _stream(stream))
    _check(code, "ep_route_topk")
    return topk_idx, topk_w
