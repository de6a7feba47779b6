"""CUDA path vs the CPU oracle, through the C ABI (needs a GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_expert_histogram_gb300 import binding as ep
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the whole module needs a device
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from combine_expert_histogram_gb300 import build as b
    b.build()


# The five workloads at full size, every token compared: all layout entries,
# every dispatched row and scale word of every (token, k), and every combined
# output element (16384 x 7168 at the DeepSeek-V3 prefill shape), in token
# chunks against the oracle.
FULL = ["tiny", "qwen3_30b_a3b_decode", "dsv3_decode", "dsv3_prefill", "skewed_zipf"]


@pytest.mark.parametrize("name", FULL)
def test_workload_parity(name):
    w = workloads.CONFIGS[name]
    case = gh.make_case(w)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    assert ref["status"] == 0
    assert gh.check_dispatch(w, case, g, ref) == w.T  # every token's rows and scales
    frac = gh.check_combine(w, case, g, ref)          # every token's output elements
    assert frac == 1.0, f"combine within 1 ulp but only {frac:.6f} bit-exact"


# Mid-size cases: several layout tiles with a ragged tail, hidden sizes whose
# UE8M0 words are partly padding, alignment 1, one hot expert, -1 ids.
MID = [
    workloads.Workload("ragged_fp8_ue8m0", T=3001, H=640, E=64, K=8, routing="softmax",
                       layout="contig", quant="fp8_ue8m0", align=128, R=4, seed=3),
    workloads.Workload("ragged_fp8_f32_masked", T=2049, H=384, E=96, K=6, routing="softmax",
                       layout="masked", quant="fp8_f32", cap=2049, seed=4),
    workloads.Workload("ragged_bf16_align1", T=1500, H=264, E=40, K=7, routing="zipf",
                       layout="contig", quant="none", align=1, R=8, seed=5),
    workloads.Workload("k32", T=600, H=1024, E=256, K=32, routing="softmax",
                       layout="contig", quant="fp8_f32", align=64, seed=6),
    workloads.Workload("k1_e1", T=777, H=256, E=1, K=1, routing="softmax",
                       layout="contig", quant="fp8_ue8m0", align=128, seed=7),
    workloads.Workload("e1024_masked", T=300, H=512, E=1024, K=4, routing="softmax",
                       layout="masked", quant="fp8_ue8m0", cap=16, R=16, seed=8),
    workloads.Workload("h128", T=5000, H=128, E=32, K=2, routing="softmax",
                       layout="contig", quant="fp8_f32", align=32, seed=9),
    # MXFP8: scale rows of 20 bytes (plain stores) and of 224 bytes (bulk stores)
    workloads.Workload("mxfp8_ragged", T=3001, H=640, E=64, K=8, routing="softmax",
                       layout="contig", quant="mxfp8", align=128, seed=12),
    workloads.Workload("mxfp8_dsv3", T=2000, H=7168, E=256, K=8, routing="grouped_sigmoid",
                       layout="masked", quant="mxfp8", cap=2000, seed=13),
    # largest hidden size: two shared-memory row stages and two output rows,
    # several slots per lane; bf16 rows of 64 KiB; and the same width through
    # the few-tokens-per-SM kernel (T <= 2 x 152)
    workloads.Workload("hmax_fp8", T=700, H=32768, E=16, K=4, routing="softmax",
                       layout="contig", quant="fp8_f32", align=16, seed=14),
    workloads.Workload("hmax_bf16", T=650, H=32768, E=16, K=4, routing="softmax",
                       layout="masked", quant="none", cap=650, seed=15),
    workloads.Workload("hmax_ue8m0_few", T=301, H=32768, E=16, K=4, routing="softmax",
                       layout="masked", quant="fp8_ue8m0", cap=301, seed=17),
    workloads.Workload("h9216_ue8m0", T=1201, H=9216, E=32, K=6, routing="softmax",
                       layout="contig", quant="fp8_ue8m0", align=64, seed=16),
    # dynamic shared memory of exactly 48 KB, which needs the limit raised
    # because the kernels also hold static shared memory (on 152 SMs): bf16
    # dispatch with 8 stages of 6 KB rows, FP8 dispatch with 2 stages + 4 rows
    # at H=6144, and the single-CTA layout at E=361
    workloads.Workload("smem48k_bf16", T=2500, H=3072, E=32, K=4, routing="softmax",
                       layout="contig", quant="none", align=64, seed=18),
    workloads.Workload("smem48k_fp8", T=400, H=6144, E=64, K=8, routing="softmax",
                       layout="contig", quant="fp8_ue8m0", align=128, seed=19),
    workloads.Workload("smem48k_layout", T=128, H=256, E=361, K=8, routing="softmax",
                       layout="contig", quant="fp8_f32", align=1, seed=20),
    # the cluster layout at its limits: K=32 (16000 entries, 16 CTAs x 4
    # rounds per warp) and E=1024 (just over 48 KB of shared memory) with a
    # masked capacity that overflows
    workloads.Workload("cluster_k32", T=500, H=256, E=256, K=32, routing="softmax",
                       layout="contig", quant="fp8_f32", align=64, seed=21),
    workloads.Workload("cluster_e1024", T=2000, H=128, E=1024, K=8, routing="zipf",
                       layout="masked", quant="fp8_ue8m0", cap=64, R=16, seed=22),
    # > 128 tiles of 2048 entries: tiles of several passes
    workloads.Workload("multipass", T=40000, H=128, E=64, K=8, routing="softmax",
                       layout="contig", quant="fp8_ue8m0", align=128, R=4, seed=10),
    workloads.Workload("multipass_e1024", T=40000, H=128, E=1024, K=8, routing="zipf",
                       layout="masked", quant="fp8_f32", cap=2048, R=8, seed=11),
]


@pytest.mark.parametrize("w", MID, ids=lambda w: w.name)
def test_mid_parity(w):
    case = gh.make_case(w)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0


def _custom_case(w, idx, wts=None):
    rng = np.random.default_rng(11)
    x = workloads.make_x(w, rng)
    if wts is None:
        wts = rng.random(idx.shape).astype(np.float32)
    return dict(idx=idx, w=wts, x=x, idx_d=torch.from_numpy(idx).cuda(),
                w_d=torch.from_numpy(wts).cuda(),
                x_d=torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))


@pytest.mark.parametrize("layout", ["contig", "masked"])
def test_single_hot_expert_and_unrouted(layout):
    """Every token on expert 3 plus -1 entries; spans several layout tiles."""
    T, K, E = 5000, 4, 16
    w = workloads.Workload("hot", T=T, H=512, E=E, K=K, routing="softmax", layout=layout,
                           quant="fp8_f32", align=128, cap=T + 5)
    idx = np.full((T, K), -1, dtype=np.int32)
    idx[:, 0] = 3
    idx[::3, 2] = 7
    case = _custom_case(w, idx)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0


def test_repeated_expert_within_token():
    """A token may name one expert twice: slots follow ascending k."""
    T, K, E = 2100, 3, 5
    w = workloads.Workload("rep", T=T, H=256, E=E, K=K, routing="softmax", layout="contig",
                           quant="none", align=4)
    idx = np.random.default_rng(2).integers(0, E, size=(T, K)).astype(np.int32)
    case = _custom_case(w, idx)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0


@pytest.mark.parametrize("T", [0, 1])
def test_tiny_token_counts(T):
    w = workloads.Workload("t", T=T, H=256, E=8, K=2, routing="softmax", layout="contig",
                           quant="fp8_ue8m0", align=128)
    idx = np.array([[5, 1]] * T, dtype=np.int32).reshape(T, 2)
    case = _custom_case(w, idx)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    gh.check_combine(w, case, g, ref)


def test_special_values_quantise_like_oracle():
    """All-zero groups, groups under the 1e-4 clamp, outliers, exact ties, -0."""
    T, H, E, K = 64, 512, 4, 2
    rng = np.random.default_rng(5)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[0] = 0.0
    xf[1] = -0.0
    xf[2] *= 1e-7
    xf[3, 5] = 3.0e38
    xf[4] = np.round(xf[4] * 8) / 8
    xf[5] *= 1e-30
    xf[6, :128] = -1e-3
    x = workloads.bf16_bits_from_f32(xf)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, K)).astype(np.float32)
    for quant in ("fp8_f32", "fp8_ue8m0", "mxfp8"):
        w = workloads.Workload("sv", T=T, H=H, E=E, K=K, routing="softmax", layout="contig",
                               quant=quant, align=16)
        case = dict(idx=idx, w=wts, x=x, idx_d=torch.from_numpy(idx).cuda(),
                    w_d=torch.from_numpy(wts).cuda(),
                    x_d=torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
        g = gh.run_gpu(w, case)
        ref = gh.check_layout(w, case, g)
        gh.check_dispatch(w, case, g, ref)


@pytest.mark.parametrize("quant", ["none", "fp8_f32", "fp8_ue8m0", "mxfp8"])
def test_masked_repack_matches_masked_dispatch(quant):
    from combine_expert_histogram_gb300 import binding as ep
    w = workloads.CONFIGS["qwen3_30b_a3b_decode"].with_(quant=quant)
    case = gh.make_case(w)
    Lc = ep.ep_layout(case["idx_d"], w.E, kind="contig", align=128)
    rows_c, sc_c, _ = ep.ep_dispatch(Lc, case["x_d"], quant)
    slab, slab_sc, mm = ep.ep_masked_repack(Lc, rows_c, sc_c, quant, w.cap)
    Lm = ep.ep_layout(case["idx_d"], w.E, kind="masked", capacity=w.cap)
    rows_m, sc_m, _ = ep.ep_dispatch(Lm, case["x_d"], quant)
    torch.cuda.synchronize()
    cnt = Lc.expert_count.cpu().numpy()
    assert np.array_equal(mm.cpu().numpy(), np.minimum(cnt, w.cap))
    assert int(Lc.status.item()) == 0
    ref = oracle.default().layout(case["idx"], w.E, "masked", cap=w.cap)
    valid = np.nonzero(ref["row_src"] >= 0)[0]
    v = torch.from_numpy(valid).cuda()
    flat = slab.reshape(w.E * w.cap, -1)
    assert torch.equal(flat.index_select(0, v).view(torch.uint8) if quant == "none" else flat.index_select(0, v),
                       rows_m.index_select(0, v).view(torch.uint8) if quant == "none" else rows_m.index_select(0, v))
    if quant != "none":
        assert torch.equal(slab_sc.reshape(w.E * w.cap, -1).index_select(0, v).view(torch.int32),
                           sc_m.index_select(0, v).view(torch.int32))


def test_masked_repack_vs_oracle_with_overflow():
    from combine_expert_histogram_gb300 import binding as ep
    w = workloads.CONFIGS["qwen3_30b_a3b_decode"]
    case = gh.make_case(w)
    cap = 12  # most experts overflow
    Lc = ep.ep_layout(case["idx_d"], w.E, kind="contig", align=128)
    rows_c, sc_c, _ = ep.ep_dispatch(Lc, case["x_d"], "fp8_f32")
    slab = torch.full((w.E, cap, w.H), gh.SENTINEL_U8, dtype=torch.uint8, device="cuda")
    slab_sc = torch.zeros((w.E, cap, w.H // 128), dtype=torch.float32, device="cuda")
    ep.ep_masked_repack(Lc, rows_c, sc_c, "fp8_f32", cap, slab=slab, slab_scales=slab_sc)
    torch.cuda.synchronize()
    orc = oracle.default()
    rows_np = rows_c.cpu().numpy()
    sc_np = sc_c.cpu().numpy()
    o_slab, o_ss, o_mm, o_st = orc.masked_repack(rows_np, sc_np, w.H, "fp8_f32",
                                                 Lc.expert_offset.cpu().numpy(),
                                                 Lc.expert_count.cpu().numpy(), w.E, cap,
                                                 fill=gh.SENTINEL_U8)
    assert o_st == 2 and int(Lc.status.item()) == 2
    assert np.array_equal(slab.reshape(w.E * cap, -1).cpu().numpy(), o_slab)
    m = np.repeat(np.arange(cap)[None, :] < o_mm[:, None], 1).reshape(-1)
    assert np.array_equal(slab_sc.reshape(w.E * cap, -1).cpu().numpy()[m], o_ss[m])


@pytest.mark.parametrize("quant", ["fp8_ue8m0", "none", "mxfp8"])
def test_dispatch_kernel_boundary(quant):
    """Dispatch picks its kernel by load: registers up to 2 tokens per SM, the
    shared-memory ring above.  Both sides of the boundary match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for T in (2 * sms, 2 * sms + 1):
        w = workloads.Workload(f"boundary_{quant}_{T}", T=T, H=7168, E=64, K=8,
                               routing="softmax", layout="masked" if quant == "fp8_ue8m0" else "contig",
                               quant=quant, align=128, cap=T, seed=T)
        case = gh.make_case(w)
        g = gh.run_gpu(w, case)
        ref = gh.check_layout(w, case, g)
        gh.check_dispatch(w, case, g, ref)
        assert gh.check_combine(w, case, g, ref) == 1.0


@pytest.mark.parametrize("K", [16, 13])  # 16-byte index loads; scalar index loads
def test_combine_cancelling_sums_bit_exact(K):
    """Entries k and k + K//2 of a token carry the same weight and opposite
    expert rows, so every sum nearly cancels and only separately rounded
    products and sums reproduce the oracle's bits; a fused multiply-add (or any
    other reordering) shows up here at once."""
    T, H, E = 2048, 1024, 64
    half = K // 2
    rng = np.random.default_rng(77)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, K)).astype(np.float32)
    wts[:, half:2 * half] = wts[:, :half]
    orc = oracle.default()
    ref = orc.layout(idx, E, "contig", align=1)
    rows, dst = ref["rows"], ref["dst_row"]
    x = rng.standard_normal((rows, H)).astype(np.float32)
    y_bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    y_bits[dst[:, half:2 * half].ravel()] = y_bits[dst[:, :half].ravel()] ^ 0x8000  # exact negation
    y = torch.from_numpy(y_bits.view(np.int16)).cuda().view(torch.bfloat16)
    L = ep.ep_layout(torch.from_numpy(idx).cuda(), E, kind="contig", align=1)
    out = ep.ep_combine(L, y, torch.from_numpy(wts).cuda())
    torch.cuda.synchronize()
    expect = orc.combine(y_bits, wts, dst, H)
    assert np.array_equal(gh.to_np_u16(out), expect)


@pytest.mark.parametrize("shift", ["dst_row", "topk_w", "y"])
def test_combine_index_arrays_not_16_byte_aligned(shift):
    """K % 4 == 0 but one index array only 4-byte aligned (combine must take
    the one-entry-at-a-time loads), or y only 16-byte aligned (the 16-byte
    lanes instead of 256-bit loads): still the oracle's bits."""
    w = workloads.Workload("align4", T=7777, H=512, E=32, K=8, routing="softmax",
                           layout="contig", quant="none", align=16, seed=23)
    case = gh.make_case(w)
    L = ep.ep_layout(case["idx_d"], w.E, kind="contig", align=w.align)
    wts = case["w_d"]
    if shift == "dst_row":
        buf = torch.empty(L.dst_row.numel() + 1, dtype=torch.int32, device="cuda")
        buf[1:].copy_(L.dst_row)
        L.dst_row = buf[1:]
    else:
        buf = torch.empty(wts.numel() + 1, dtype=torch.float32, device="cuda")
        buf[1:].copy_(wts.view(-1))
        wts = buf[1:].view(wts.shape)
    y = workloads.make_expert_outputs(L.rows_capacity, w.H, seed=3, device="cuda")
    if shift == "y":  # same values, 16 bytes past a 32-byte boundary
        buf = torch.empty(y.numel() + 8, dtype=torch.bfloat16, device="cuda")
        buf[8:].copy_(y.view(-1))
        y = buf[8:].view(y.shape)
        assert y.data_ptr() % 32 == 16
    out = ep.ep_combine(L, y, wts)
    torch.cuda.synchronize()
    ref = oracle.default().layout(case["idx"], w.E, "contig", align=w.align)
    dst = ref["dst_row"]
    y_bits = gh.to_np_u16(y)
    expect = oracle.default().combine(y_bits, case["w"], dst, w.H)
    assert np.array_equal(gh.to_np_u16(out), expect)


# row_src is optional: without it the cluster kernel runs one cluster with no
# fill, and the tiled kernels no fill CTAs; every other array must be the same
@pytest.mark.parametrize("name,T", [("qwen3_30b_a3b_decode", None), ("dsv3_decode", None),
                                    ("skewed_zipf", 1500), ("dsv3_prefill", 3000)])
def test_layout_without_row_src(name, T):
    w = workloads.CONFIGS[name]
    if T is not None:
        w = w.with_(T=T, name=f"{name}_T{T}")
    case = gh.make_case(w)
    g = gh.run_gpu(w, case, with_row_src=False)
    assert g["L"].row_src is None
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0


# rank_rows is optional as well (alone, and with row_src also absent)
@pytest.mark.parametrize("T,layout,no_row_src", [(256, "masked", False), (256, "masked", True),
                                                 (3000, "contig", False), (3000, "contig", True),
                                                 (3000, "masked", False), (3000, "masked", True)])
def test_layout_without_rank_rows(T, layout, no_row_src):
    w = workloads.CONFIGS["skewed_zipf"].with_(T=T, H=128, layout=layout, cap=T,
                                               name=f"no_rank_rows_{T}_{layout}")
    case = gh.make_case(w)
    L = ep.new_layout(w.T, w.K, w.E, w.layout, align=w.align, capacity=w.cap, num_ranks=w.R,
                      with_row_src=not no_row_src)
    L.rank_rows = None
    L.status.fill_(7)
    ep.ep_layout(case["idx_d"], w.E, out=L)
    torch.cuda.synchronize()
    ref = oracle.default().layout(case["idx"], w.E, w.layout, align=w.align, cap=w.cap, R=w.R)
    assert int(L.status.item()) == ref["status"]
    assert np.array_equal(L.expert_count.cpu().numpy(), ref["count"])
    assert np.array_equal(L.expert_offset.cpu().numpy(), ref["offset"])
    assert np.array_equal(L.dst_row.cpu().numpy().reshape(w.T, w.K), ref["dst_row"])
    if L.row_src is not None:
        assert np.array_equal(L.row_src.cpu().numpy()[:ref["rows"]], ref["row_src"])


# A large layout on the tiled path: 800000 entries at E = 1024, so 98 tiles
# of four passes each (a histogram kernel and an assign kernel), contiguous
# and masked (with row_src, so with fill CTAs)
@pytest.mark.parametrize("layout", ["contig", "masked"])
def test_tiled_layout_with_passes(layout):
    w = workloads.Workload(f"tiled_{layout}", T=100000, H=128, E=1024, K=8, routing="softmax",
                           layout=layout, quant="fp8_f32", align=128, cap=900, R=8, seed=31)
    idx = np.random.default_rng(31).integers(-1, w.E, size=(w.T, w.K)).astype(np.int32)
    case = _custom_case(w, idx)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref, sample_tokens=2048)
    assert gh.check_combine(w, case, g, ref, sample_tokens=2048) == 1.0


# The two sides of the decode layout's limit: 16384 entries (the largest
# cluster launch: 16 CTAs of 4 rounds per warp, with counting clusters) and
# 16385 (the first tiled launch), masked with row_src and contiguous
@pytest.mark.parametrize("T,K,layout", [(2048, 8, "masked"), (2048, 8, "contig"),
                                        (3277, 5, "masked"), (3277, 5, "contig")])
def test_layout_at_the_cluster_limit(T, K, layout):
    w = workloads.Workload(f"limit_{T * K}_{layout}", T=T, H=256, E=96, K=K, routing="softmax",
                           layout=layout, quant="fp8_ue8m0", align=64, cap=T, R=4, seed=51)
    idx = np.random.default_rng(51 + T * K).integers(-1, w.E, size=(T, K)).astype(np.int32)
    case = _custom_case(w, idx)
    g = gh.run_gpu(w, case)
    ref = gh.check_layout(w, case, g)
    gh.check_dispatch(w, case, g, ref)
    assert gh.check_combine(w, case, g, ref) == 1.0
