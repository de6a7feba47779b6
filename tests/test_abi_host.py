"""The C-ABI library builds, loads and exports every symbol include/ep.h declares;
host-side argument validation (no GPU needed: it returns before any CUDA call)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from combine_expert_histogram_gb300 import build as b
    if not b.up_to_date():
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libep.so")
        b.build()
    from combine_expert_histogram_gb300 import binding
    return binding.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) >= {"ep_layout", "ep_dispatch", "ep_combine", "ep_masked_repack"}
    for n in names:
        assert hasattr(lib, n), f"libep.so does not export {n}"
    from combine_expert_histogram_gb300 import binding
    assert set(binding.EXPORTS) >= set(names)


def _layout(**kw):
    from combine_expert_histogram_gb300.binding import _Layout
    c = _Layout()
    d = dict(num_tokens=16, num_topk=8, num_experts=256, num_ranks=1, kind=0, align=128,
             capacity=0, max_tokens=0)
    d.update(kw)
    for k, v in d.items():
        setattr(c, k, v)
    return c


def test_sizing_helpers(lib):
    assert lib.ep_rows_capacity(ctypes.byref(_layout())) == 16 * 8 + 128 * 127
    assert lib.ep_rows_capacity(ctypes.byref(_layout(num_tokens=16384))) == 16384 * 8 + 256 * 127
    assert lib.ep_rows_capacity(ctypes.byref(_layout(kind=1, capacity=1024))) == 256 * 1024
    assert lib.ep_rows_capacity(ctypes.byref(_layout(num_topk=33))) == -1
    assert lib.ep_rows_capacity(ctypes.byref(_layout(align=96))) == -1
    assert lib.ep_rows_capacity(ctypes.byref(_layout(num_experts=1025))) == -1
    assert lib.ep_rows_capacity(ctypes.byref(_layout(num_ranks=3))) == -1
    assert lib.ep_scale_cols(7168, 1) == 56
    assert lib.ep_scale_cols(7168, 2) == 14
    assert lib.ep_scale_cols(384, 2) == 1
    assert lib.ep_scale_cols(2048, 0) == 0
    assert lib.ep_scale_cols(200, 1) == -1
    # hidden sizes up to EP_MAX_HIDDEN = 32768 (rows are staged in shared memory)
    assert lib.ep_scale_cols(32768, 1) == 256
    assert lib.ep_scale_cols(32768 + 128, 1) == -1
    # up to 16384 entries one kernel of one thread-block cluster and no scratch;
    # beyond, tiles of 1024 entries (2048 above 32768 entries) need tiles x E int32
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=0))) == 0
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=128))) == 0
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=1024))) == 0
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=2048))) == 0
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=2049))) == 17 * 256 * 4
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=4096))) == 32 * 256 * 4
    assert lib.ep_layout_workspace_bytes(ctypes.byref(_layout(num_tokens=16384))) == 64 * 256 * 4


def test_host_validation_returns_before_any_launch(lib):
    INVALID, CAPACITY = 1, 2
    L = _layout()
    # NULL layout arrays
    assert lib.ep_layout(None, ctypes.byref(L), None, 0, None) == INVALID
    L.dst_row = L.expert_count = L.expert_offset = L.status = 256
    # NULL topk_idx with tokens present
    assert lib.ep_layout(None, ctypes.byref(L), None, 0, None) == INVALID
    # too many tokens for the reserved capacity: fail fast with an error code
    L.max_tokens = 8
    assert lib.ep_layout(ctypes.c_void_p(4096), ctypes.byref(L), None, 0, None) == CAPACITY
    L.max_tokens = 0
    # K beyond the top-32 limit
    L.num_topk = 33
    assert lib.ep_layout(ctypes.c_void_p(4096), ctypes.byref(L), None, 0, None) == INVALID
    L.num_topk = 8
    # misaligned x / rows, bad hidden, unpaired topk_w / row_w
    assert lib.ep_dispatch(ctypes.byref(L), ctypes.c_void_p(4100), 7168, 1, ctypes.c_void_p(4096),
                           ctypes.c_void_p(4096), None, None, None) == INVALID
    assert lib.ep_dispatch(ctypes.byref(L), ctypes.c_void_p(4096), 7000, 1, ctypes.c_void_p(4096),
                           ctypes.c_void_p(4096), None, None, None) == INVALID
    assert lib.ep_dispatch(ctypes.byref(L), ctypes.c_void_p(4096), 7168, 1, ctypes.c_void_p(4096),
                           None, None, None, None) == INVALID
    assert lib.ep_dispatch(ctypes.byref(L), ctypes.c_void_p(4096), 7168, 0, ctypes.c_void_p(4096),
                           None, ctypes.c_void_p(4096), None, None) == INVALID
    assert lib.ep_combine(ctypes.byref(L), ctypes.c_void_p(4104), 7168, ctypes.c_void_p(4096),
                          ctypes.c_void_p(4096), None) == INVALID
    # repack needs a contiguous layout and a positive capacity
    Lm = _layout(kind=1, capacity=64)
    Lm.dst_row = Lm.expert_count = Lm.expert_offset = Lm.status = 256
    assert lib.ep_masked_repack(ctypes.byref(Lm), ctypes.c_void_p(4096), None, 7168, 0, 64,
                                ctypes.c_void_p(4096), None, ctypes.c_void_p(4096), None) == INVALID
    assert lib.ep_masked_repack(ctypes.byref(L), ctypes.c_void_p(4096), None, 7168, 0, 0,
                                ctypes.c_void_p(4096), None, ctypes.c_void_p(4096), None) == INVALID
    assert lib.ep_dispatch(ctypes.byref(L), ctypes.c_void_p(4096), 32776, 0, ctypes.c_void_p(4096),
                           None, None, None, None) == INVALID
    assert lib.ep_status_str(3).decode().startswith("EP_ERR_BAD_EXPERT_ID")
    assert lib.ep_status_str(6).decode().startswith("EP_ERR_TIMEOUT")


def test_noalloc_checks_arguments_before_its_scratch_size(lib):
    """ep_layout_noalloc gives ep_layout's code for bad arguments even on a
    shape too large for its fixed array, and EP_ERR_CAPACITY only for a
    well-formed call; all before any CUDA call."""
    INVALID, CAPACITY = 1, 2
    from combine_expert_histogram_gb300 import binding
    L = _layout(num_tokens=70000, num_experts=1024)
    assert lib.ep_layout_workspace_bytes(ctypes.byref(L)) > binding.NOALLOC_SCRATCH_BYTES
    assert lib.ep_layout_noalloc(ctypes.c_void_p(4096), ctypes.byref(L), None) == INVALID
    L.dst_row = L.expert_count = L.expert_offset = L.status = 256
    assert lib.ep_layout_noalloc(None, ctypes.byref(L), None) == INVALID
    assert lib.ep_layout_noalloc(ctypes.c_void_p(4098), ctypes.byref(L), None) == INVALID
    L.max_tokens = 8
    assert lib.ep_layout_noalloc(ctypes.c_void_p(4096), ctypes.byref(L), None) == CAPACITY
    L.max_tokens = 0
    assert lib.ep_layout_noalloc(ctypes.c_void_p(4096), ctypes.byref(L), None) == CAPACITY
    assert lib.ep_layout_noalloc(ctypes.c_void_p(4096), None, None) == INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from combine_expert_histogram_gb300 import binding
    with pytest.raises(ValueError):
        binding._ptr(torch.zeros(4, dtype=torch.int32))


def test_nvtx_ranges_around_a_call_that_returns_early(lib):
    """EP_NVTX=1: the range around an entry point is pushed and popped also
    when the call returns an argument error (no GPU needed)."""
    import subprocess
    import sys
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    child = ("import sys, ctypes; sys.path.insert(0, %r)\n"
             "from combine_expert_histogram_gb300 import binding as b\n"
             "lib = b.load_library()\n"
             "L = b._Layout(); L.num_tokens = 4; L.num_topk = 2; L.num_experts = 8\n"
             "L.num_ranks = 1; L.align = 1\n"
             "assert lib.ep_layout(None, ctypes.byref(L), None, 0, None) == 1\n"
             "assert lib.ep_combine(None, None, 128, None, None, None) == 1\n"
             "print('ok')\n" % root)
    r = subprocess.run([sys.executable, "-c", child], env=dict(os.environ, EP_NVTX="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
