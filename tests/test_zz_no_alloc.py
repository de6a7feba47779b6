"""ep_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (runtimes that reserve all memory at start-up, plugins handed only
their input and output buffers).  It takes its scratch from a fixed array in the
library; its results must equal ep_layout's with a caller-provided workspace.

Collected last on purpose; it also passes when run alone in a fresh process.
"""
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


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, K, E = 70000, 8, 1024  # 69 tiles x 1024 experts x 4 B > 256 KiB
    L = ep.new_layout(T, K, E, "contig", align=128)
    assert ep.ep_layout_workspace_bytes(L) > ep.NOALLOC_SCRATCH_BYTES
    idx = torch.zeros(T, K, dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EPError) as ei:
        ep.ep_layout_noalloc(idx, L)
    assert ei.value.code == ep.EP_ERR_CAPACITY
