"""The bench's host-side bookkeeping on CPU: algorithmic bytes, the e2e run's
host pool plan and the digest-keyed ncu traffic lookup."""

from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import WORKLOADS  # noqa: E402

W = WORKLOADS["qwen3_4b_b192"]
HEADS_TOTAL = W.layers * W.batch * W.heads  # 221,184 query heads


def test_score_bytes_per_unit_follow_the_definition():
    # per unit with nothing moved: K read once (2064 x 256 B) + 128 observation
    # rows (128 x 256 B) + 2048 kept indices (x 4 B) = 569,344 bytes
    kb = bench.kernel_bytes(W, R=128, rows_moved_per_launch=0, heads_total=HEADS_TOTAL, n_fps=32)
    assert W.units == 55_296
    assert kb["score_select"] == 55_296 * 569_344
    # each moved row adds its V read and its K and V writes: 3 x 256 bytes
    kb1 = bench.kernel_bytes(W, R=128, rows_moved_per_launch=1000, heads_total=HEADS_TOTAL, n_fps=32)
    assert kb1["score_select"] - kb["score_select"] == 768_000
    # FPS reads 32 candidate rows and writes 16 beacons (+1 trace byte each) per head
    assert kb["fps"] == HEADS_TOTAL * (32 * 256 + 16 * 257)
    assert kb["append"] == HEADS_TOTAL * 512


def test_step_bytes_match_the_stated_113_gb():
    # 1,863.29 rows moved per unit: one step (eviction + 16 appends) moves
    # 113.33 GB algorithmic, the figure quoted for this workload
    m_unit = 1863.2923538773148
    got = bench.path_bytes(W, R=128, rows_moved_per_eviction=m_unit * W.units, heads_total=HEADS_TOTAL)
    assert abs(got - 113_329_402_368) < 1e3


def test_e2e_plan_keeps_every_period_distinct_within_the_host_cap():
    cap = 48 << 30
    default_period = 16 * 36 * 192 * 32 * 128 * 2   # 0.91 GB of queries per period
    sched_period = 256 * 36 * 192 * 32 * 128 * 2    # 14.5 GB per period (7/8 schedule)
    assert bench.e2e_plan(default_period, 3, 10, cap) == (3, 10)
    assert bench.e2e_plan(default_period, 0, 10, cap) == (1, 10)  # at least one warm-up step
    # three periods fit in 48 GB: one warm-up and two timed steps
    assert bench.e2e_plan(sched_period, 3, 5, cap) == (1, 2)
    # a period larger than the cap still runs one warm-up and one timed step
    assert bench.e2e_plan(cap + 1, 3, 5, cap) == (1, 1)
    for per in (default_period, sched_period, cap // 3 + 1):
        warm, timed = bench.e2e_plan(per, 3, 10, cap)
        assert warm >= 1 and timed >= 1
        assert (warm + timed) * per <= max(cap, 2 * per)


def test_traffic_row_applies_only_to_its_source_digest(monkeypatch):
    real = bench.kernel_source_digest("score_select")
    assert real and len(real) == 16
    got = bench.read_traffic("score_select", "qwen3_4b_b192")
    # the committed table lists the current source, or the lookup declines
    if got is not None:
        assert got > 0
    assert bench.read_traffic("score_select", "no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_digest", lambda kernel: "0" * 16)
    assert bench.read_traffic("score_select", "qwen3_4b_b192") is None
    assert bench.read_traffic("rope", "qwen3_4b_b192") is None
