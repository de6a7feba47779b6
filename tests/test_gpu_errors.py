"""Error paths on the GPU: data-dependent errors land in the status word, never
as a trap, a hang or an out-of-bounds write (guard bands around every output
are checked).  Host-detectable errors return before any launch."""
import numpy as np
import pytest
import torch

import oracle
from combine_expert_histogram_gb300 import binding as ep

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

GUARD = 4096
PAT = 0x5A5A5A5A  # int32 guard pattern


def _guarded(n, dtype=torch.int32):
    buf = torch.full((n + 2 * GUARD,), PAT, dtype=torch.int32, device="cuda")
    return buf, buf[GUARD:GUARD + n]


def _guards_intact(buf, n):
    return bool((buf[:GUARD] == PAT).all()) and bool((buf[GUARD + n:] == PAT).all())


# cluster kernel of 1, 8 and 16 CTAs (4 rounds per warp); histogram + assign kernels
@pytest.mark.parametrize("T", [50, 500, 3000, 5000])
def test_bad_expert_ids_raise_status_without_stray_writes(T):
    E, K = 16, 4
    rng = np.random.default_rng(0)
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[3, 1] = E
    idx[7, 0] = -5
    idx[T - 1, 3] = 1 << 30
    L = ep.new_layout(T, K, E, "contig", align=8)
    rows = L.rows_capacity
    rs_buf, L.row_src = _guarded(rows)
    dr_buf, L.dst_row = _guarded(T * K)
    ep.ep_layout(torch.from_numpy(idx).cuda(), E, out=L)
    torch.cuda.synchronize()
    assert int(L.status.item()) == ep.EP_ERR_BAD_EXPERT_ID
    with pytest.raises(ep.EPError):
        L.check_status()
    ref = oracle.default().layout(idx, E, "contig", align=8)
    assert ref["status"] == 3
    assert np.array_equal(L.dst_row.cpu().numpy().reshape(T, K), ref["dst_row"])
    assert np.array_equal(L.row_src.cpu().numpy()[:ref["rows"]], ref["row_src"])
    assert _guards_intact(rs_buf, rows) and _guards_intact(dr_buf, T * K)


@pytest.mark.parametrize("T", [40, 700, 4000, 4500])
def test_masked_capacity_overflow(T):
    E, K, cap = 8, 4, 9
    rng = np.random.default_rng(1)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    L = ep.new_layout(T, K, E, "masked", capacity=cap)
    rows = E * cap
    rs_buf, L.row_src = _guarded(rows)
    ep.ep_layout(torch.from_numpy(idx).cuda(), E, kind="masked", capacity=cap, out=L)
    x = torch.randn(T, 256, device="cuda").to(torch.bfloat16)
    out_buf = torch.full(((rows + 8) * 256,), 0x5A, dtype=torch.uint8, device="cuda")
    out_rows = out_buf[4 * 256:(rows + 4) * 256].view(rows, 256)
    sc = torch.zeros(rows, 2, dtype=torch.float32, device="cuda")
    ep.ep_dispatch(L, x, "fp8_f32", out_rows=out_rows, out_scales=sc)
    torch.cuda.synchronize()
    assert int(L.status.item()) == ep.EP_ERR_CAPACITY
    ref = oracle.default().layout(idx, E, "masked", cap=cap)
    assert ref["status"] == 2
    assert np.array_equal(L.dst_row.cpu().numpy().reshape(T, K), ref["dst_row"])
    assert np.array_equal(L.expert_count.cpu().numpy(), ref["count"])
    assert _guards_intact(rs_buf, rows)
    assert bool((out_buf[:4 * 256] == 0x5A).all()) and bool((out_buf[(rows + 4) * 256:] == 0x5A).all())


def test_token_capacity_is_checked_before_launch():
    idx = torch.zeros(200, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EPError) as ei:
        ep.ep_layout(idx, 16, max_tokens=128)
    assert ei.value.code == ep.EP_ERR_CAPACITY


def test_status_resets_on_next_layout():
    E = 4
    bad = torch.tensor([[0, 9]], dtype=torch.int32, device="cuda")
    L = ep.ep_layout(bad, E, align=4)
    torch.cuda.synchronize()
    assert int(L.status.item()) == ep.EP_ERR_BAD_EXPERT_ID
    good = torch.tensor([[0, 3]], dtype=torch.int32, device="cuda")
    ep.ep_layout(good, E, align=4, out=L)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0


@pytest.mark.parametrize("T", [300, 3000])  # cluster kernel; histogram + assign kernels
def test_multi_tile_status_max_and_reset(T):
    """Bad ids and an over-full masked expert together report the larger code;
    the next layout of good ids resets it."""
    E, K, cap = 16, 8, 8
    rng = np.random.default_rng(2)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[T // 2, 5] = E + 3
    L = ep.new_layout(T, K, E, "masked", capacity=cap)
    ep.ep_layout(torch.from_numpy(idx).cuda(), E, kind="masked", capacity=cap, out=L)
    torch.cuda.synchronize()
    ref = oracle.default().layout(idx, E, "masked", cap=cap)
    assert int(L.status.item()) == ref["status"] == ep.EP_ERR_BAD_EXPERT_ID
    assert np.array_equal(L.dst_row.cpu().numpy().reshape(T, K), ref["dst_row"])
    good = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    L2 = ep.new_layout(T, K, E, "masked", capacity=T)
    L2.status = L.status  # the status word still holds the error
    ep.ep_layout(torch.from_numpy(good).cuda(), E, kind="masked", capacity=T, out=L2)
    torch.cuda.synchronize()
    assert int(L2.status.item()) == 0


# cluster kernel of 1-2 and 13 CTAs; histogram + assign kernels
@pytest.mark.parametrize("cap", [64, 800, 5000])
def test_masked_capacity_exact_boundary(cap):
    """An expert receiving exactly `capacity` rows is fine; one row more raises
    EP_ERR_CAPACITY and only the extra entry goes unplaced."""
    E, K = 16, 4
    rng = np.random.default_rng(cap)
    for extra in (0, 1):
        T = cap + extra
        idx = np.stack([np.concatenate([[0], 1 + rng.permutation(E - 1)[:K - 1]])
                        for _ in range(T)]).astype(np.int32)  # expert 0 in every token
        L = ep.new_layout(T, K, E, "masked", capacity=cap)
        ep.ep_layout(torch.from_numpy(idx).cuda(), E, kind="masked", capacity=cap, out=L)
        torch.cuda.synchronize()
        ref = oracle.default().layout(idx, E, "masked", cap=cap)
        assert int(L.status.item()) == ref["status"] == (ep.EP_ERR_CAPACITY if extra else 0)
        got = L.dst_row.cpu().numpy().reshape(T, K)
        assert np.array_equal(got, ref["dst_row"])
        assert int((got[:, 0] < 0).sum()) == extra  # only the last token's expert-0 entry
        assert int(L.expert_count.cpu()[0]) == T


def test_bounded_wait_gives_up_and_reports():
    """The dispatch kernels' mbarrier waits are bounded: a wait on a barrier
    that nothing completes returns after its limit and raises EP_ERR_TIMEOUT
    into the status word, and the context stays usable."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_selftest_bounded_wait(status, 1 << 20)  # about half a millisecond
    torch.cuda.synchronize()
    assert int(status.item()) == ep.EP_ERR_TIMEOUT
    # the GPU still runs work afterwards
    idx = torch.tensor([[0, 3], [1, 2], [3, 0]], dtype=torch.int32, device="cuda")
    L = ep.ep_layout(idx, 4, align=4)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    ref = oracle.default().layout(idx.cpu().numpy(), 4, "contig", align=4)
    assert L.dst_row.cpu().tolist() == ref["dst_row"].ravel().tolist()
    with pytest.raises(ep.EPError):
        ep.ep_selftest_bounded_wait(status, 0)  # limits outside 1 .. 2^31 are refused


def test_cluster_bounded_wait_gives_up_and_reports():
    """The decode layout's histogram exchange waits on a barrier for its
    peers' bulk copies; that wait is bounded too: in a 2-CTA cluster whose
    peers send nothing, both waits give up, the CTAs still meet at the
    closing cluster barrier, EP_ERR_TIMEOUT lands in the status word, and the
    context stays usable (a cluster layout runs and matches the oracle)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_selftest_cluster_wait(status, 1 << 20)
    torch.cuda.synchronize()
    assert int(status.item()) == ep.EP_ERR_TIMEOUT
    rng = np.random.default_rng(4)
    idx = rng.integers(0, 64, size=(300, 8)).astype(np.int32)  # 2400 entries: cluster path
    L = ep.ep_layout(torch.from_numpy(idx).cuda(), 64, kind="masked", capacity=300)
    torch.cuda.synchronize()
    ref = oracle.default().layout(idx, 64, "masked", cap=300)
    assert int(L.status.item()) == ref["status"] == 0
    assert np.array_equal(L.dst_row.cpu().numpy().reshape(idx.shape), ref["dst_row"])
    with pytest.raises(ep.EPError):
        ep.ep_selftest_cluster_wait(status, (1 << 31) + 1)
