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
