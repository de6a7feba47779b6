"""bench.py's host-side accounting (no GPU): the algorithmic bytes behind every
GB/s and roofline fraction equal the survey's per-token table for the five
workloads, and the replica arithmetic of the whole-job value."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

# bytes per token the method must move (dispatch, combine): 2H (x) + 4K
# (dst_row) + K rows; K x 2H (y) + 4K (w) + 4K (dst_row) + 2H (out)
PER_TOKEN = {
    "tiny": (1544, 1552),
    "qwen3_30b_a3b_decode": (21024, 36928),
    "dsv3_decode": (72160, 129088),
    "dsv3_prefill": (73504, 129088),
    "skewed_zipf": (73760, 73792),
}


@pytest.mark.parametrize("name", list(PER_TOKEN))
def test_algorithmic_bytes_per_token(name):
    w = workloads.CONFIGS[name]
    ab = bench.algorithmic_bytes(w)
    disp, comb = PER_TOKEN[name]
    assert ab["dispatch"] == disp * w.T
    assert ab["combine"] == comb * w.T
    assert ab["layout"] == 12 * w.K * w.T  # idx read, dst_row and row_src written


def test_prefill_launch_bytes():
    w = workloads.CONFIGS["dsv3_prefill"]
    ab = bench.algorithmic_bytes(w)
    assert ab["dispatch"] == 1_204_289_536
    assert ab["combine"] == 2_114_977_792


def test_whole_job_tokens_per_s():
    # 4 replicas of 16384 tokens, 10 steps, slowest rank 5.0 ms in all
    assert bench.aggregate_tokens_per_s(16384, 10, 4, 5.0) == pytest.approx(16384 * 10 * 4 / 5e-3)


def test_print_table_on_full_and_partial_lines():
    """The stderr summary handles the fields a line may lack (no decode
    section, no CPU baseline, kernels without a token rate)."""
    import io
    full = {"config": {"workload": "dsv3_prefill", "T": 16384, "H": 7168, "E": 256, "K": 8,
                       "quant": "fp8_f32"},
            "ms_per_step": 0.51, "value": 3.2e7, "step_gbs": 6500.0,
            "roofline": {"peak": 6694.8, "peak_source": "measured"},
            "kernels": {"layout": {"us": 14.2, "GB/s": 110.0, "frac_of_peak": 0.016},
                        "combine": {"us": 309.0, "GB/s": 6840.0, "frac_of_peak": 1.02}},
            "decode": {"qwen3_30b_a3b_decode": {"step_us_graph": 6.8,
                                                "from_logits": {"step_us_graph": 8.7},
                                                "warm_graph_us": {"layout": 2.7}}},
            "cpu_baseline": {"value": 6000.0, "cores": 1},
            "e2e": {"value": 1.3e6}}
    buf = io.StringIO()
    bench.print_table(full, out=buf)
    text = buf.getvalue()
    assert "dsv3_prefill" in text and "combine" in text and "from logits 8.7" in text
    assert "CPU oracle (1 core)" in text and "end to end" in text
    buf = io.StringIO()
    bench.print_table({"config": {"workload": "tiny"}, "kernels": {"layout": {}}}, out=buf)
    assert "tiny" in buf.getvalue()
