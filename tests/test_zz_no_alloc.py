"""ep_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (runtimes that reserve all memory at start-up, plugins handed only
their input and output buffers).  It takes its scratch from a fixed array in the
library; its results must equal ep_layout's with a caller-provided workspace.

Collected last on purpose; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from combine_expert_histogram_gb300 import binding as ep

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from combine_expert_histogram_gb300 import build as b
    b.build()


def _fields(L):
    T, K = L.num_tokens, L.num_topk
    rows = int(L.expert_offset[-1].item())
    return dict(dst_row=L.dst_row[:T * K].cpu().numpy(),
                row_src=L.row_src[:rows].cpu().numpy(),
                count=L.expert_count.cpu().numpy(),
                offset=L.expert_offset.cpu().numpy(),
                rank_rows=L.rank_rows.cpu().numpy(),
                status=int(L.status.item()))


def _layouts_equal(a, b):
    fa, fb = _fields(a), _fields(b)
    for k in fa:
        assert np.array_equal(fa[k], fb[k]), f"{k} differs"


def test_noalloc_matches_ep_layout_on_two_calls_in_a_row():
    # two different multi-tile shapes back to back: the shared scratch array
    # must carry nothing from the first call into the second
    for name in ("dsv3_prefill", "skewed_zipf"):
        w = workloads.CONFIGS[name]
        idx, _, _ = workloads.make_inputs(w)
        idx_d = torch.from_numpy(idx).cuda()
        ref = ep.ep_layout(idx_d, w.E, kind=w.layout, align=w.align, capacity=w.cap,
                           num_ranks=w.R)
        assert ep.ep_layout_workspace_bytes(ref) > 0  # the shape really uses scratch
        out = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap,
                            num_ranks=w.R)
        out.workspace = None  # the no-alloc call never sees a workspace
        ep.ep_layout_noalloc(idx_d, out)
        torch.cuda.synchronize()
        _layouts_equal(out, ref)


@pytest.mark.parametrize("cap,plant", [(4096, None), (90, "capacity"), (4096, "bad_id"),
                                       (90, "both")])
def test_noalloc_masked_and_status_errors(cap, plant):
    """A masked multi-tile layout with row_src (its fill CTAs read the shared
    array too), and data-dependent errors raised after the array is used: an
    over-full expert, an id outside [-1, E), or both.  Every field, the status
    word included, equals ep_layout with a caller workspace."""
    T, K, E = 4096, 8, 256
    w = workloads.Workload("noalloc_masked", T=T, H=128, E=E, K=K, routing="softmax",
                           layout="masked", quant="none", cap=cap, R=8, seed=41)
    idx, _, _ = workloads.make_inputs(w)
    idx = idx.copy()
    if plant in ("bad_id", "both"):
        idx[1234, 3] = E + 7
        idx[4000, 0] = -5
    idx[::5, 7] = -1  # unrouted entries
    idx_d = torch.from_numpy(idx).cuda()
    ref = ep.ep_layout(idx_d, E, kind="masked", capacity=cap, num_ranks=w.R)
    assert ep.ep_layout_workspace_bytes(ref) > 0  # the shape really uses scratch
    out = ep.new_layout(T, K, E, "masked", capacity=cap, num_ranks=w.R)
    out.workspace = None
    out.status.fill_(0)
    ep.ep_layout_noalloc(idx_d, out)
    torch.cuda.synchronize()
    _layouts_equal(out, ref)
    want = {None: ep.EP_OK, "capacity": ep.EP_ERR_CAPACITY, "bad_id": ep.EP_ERR_BAD_EXPERT_ID,
            "both": ep.EP_ERR_BAD_EXPERT_ID}[plant]
    assert int(out.status.item()) == want


def test_noalloc_argument_errors_match_ep_layout():
    """Bad arguments give ep_layout's code even when the shape is also too
    large for the fixed array: argument checks come first."""
    T, K, E = 100000, 8, 1024  # per-tile histograms: 98 tiles x 1024 experts x 4 B
    L = ep.new_layout(T, K, E, "contig", align=128)
    assert ep.ep_layout_workspace_bytes(L) > ep.NOALLOC_SCRATCH_BYTES
    lib = ep.load_library()
    st = L.struct()
    # NULL topk_idx with tokens to lay out: both calls give the argument error
    assert lib.ep_layout_noalloc(None, ctypes.byref(st), None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_layout(None, ctypes.byref(st), None, 0, None) == ep.EP_ERR_INVALID_ARG


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, K, E = 100000, 8, 1024  # 98 tiles x 1024 experts x 4 B > 256 KiB
    L = ep.new_layout(T, K, E, "contig", align=128)
    assert ep.ep_layout_workspace_bytes(L) > ep.NOALLOC_SCRATCH_BYTES
    idx = torch.zeros(T, K, dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EPError) as ei:
        ep.ep_layout_noalloc(idx, L)
    assert ei.value.code == ep.EP_ERR_CAPACITY
