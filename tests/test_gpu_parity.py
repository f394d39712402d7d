"""GPU parity of the CUDA library against the CPU oracle, through the C ABI.

Each case runs a seeded synthetic stream through both sides in lockstep
(tests/lockstep.py states the agreement rules) and at sizes the oracle
finishes in seconds: several 128-key tiles plus a ragged tail, every
observation-row count the configs reach, zero beacons, short and long
periods, GQA groups 1..8, and inputs that drive FPS through its wide-exponent
exact-sum path.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from synth import WORKLOADS
from tests.lockstep import run_lockstep, run_lockstep_parallel

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_eviction_head_gb300.build import build
    build()


def assert_clean(rep, min_evictions=1):
    assert not rep.failures, "\n".join(rep.failures)
    assert rep.evictions >= min_evictions
    assert rep.units_checked >= rep.evictions


def test_tiny_full_stream():
    rep = run_lockstep(TINY, seed=0xBEAC0)
    assert_clean(rep, min_evictions=24)
    assert rep.fps_heads_checked == 4 * rep.evictions


@pytest.mark.parametrize("name,over", [
    ("zero_beacons", dict(fps_cap=16, fps_keep=0)),
    ("short_period", dict(period=8)),
    ("long_period", dict(period=24)),
    ("no_prefix_no_recent", dict(prefix=0, recent=0)),
    ("gqa1", dict(heads=1, kv_heads=1)),
    ("gqa7", dict(heads=7, kv_heads=1)),
    ("gqa8_two_kv", dict(heads=16, kv_heads=2)),
    ("ragged_budget", dict(budget=200, steps=300)),
    ("small_buffer", dict(fps_cap=6, fps_keep=2)),
    ("batch_layers", dict(layers=2, batch=3, heads=8, kv_heads=2, steps=200)),
    # 5 heads x (12..31 beacons + 16 recents): observation rows sweep 140..235,
    # so the second M tile starts at every 16-row offset past 128 (a split warp)
    ("gqa5_rows_sweep", dict(heads=5, kv_heads=1, fps_keep=12, steps=400)),
    # 224 rows and a 1016-slot cache: the single-chunk plan leaves two
    # compaction buffers, so the rows are scored in two chunks of 112
    ("gqa7_two_row_chunks", dict(heads=7, kv_heads=1, budget=1000, steps=1100)),
])
def test_tiny_variants(name, over):
    w = TINY.with_(**{"steps": 240, **over})
    rep = run_lockstep(w, seed=0xBEAC0 + len(name))
    assert_clean(rep)


@pytest.mark.parametrize("order_free", [False, True])
def test_odd_drop_count(order_free):
    """17 drops per unit (period 17): odd drop counts, which shift the shared
    memory that follows the drop lists by 8 bytes."""
    w = TINY.with_(period=17, steps=260)
    rep = run_lockstep(w, seed=0xBEAB6, order_free=order_free)
    assert_clean(rep, min_evictions=5)


def test_period_one_drops_one_slot_per_step():
    """An eviction after every append: L = budget + 1, one slot dropped, FPS over
    the beacons and a single recent query each time."""
    w = TINY.with_(period=1, steps=200)
    rep = run_lockstep(w, seed=0xBEAB7)
    assert_clean(rep, min_evictions=60)


@pytest.mark.parametrize("budget,period", [(8176, 16), (7680, 512)])
def test_longest_cache_8192_slots(budget, period):
    """The longest cache the kernels take (L = 8192: 64 tiles, the selector's
    8192-bit drop mask; the shared-memory plan falls back to fewer compaction
    chunks), with 16 drops per unit (per-lane lists) and with 512 (radix)."""
    w = TINY.with_(budget=budget, period=period, steps=8192 + 2 * period)
    rep = run_lockstep(w, seed=0xBEAB8 + period)
    assert_clean(rep, min_evictions=2)


def test_many_tiles():
    w = TINY.with_(budget=1000, steps=1100, heads=8, kv_heads=2)
    rep = run_lockstep(w, seed=7)
    assert_clean(rep, min_evictions=6)


def test_qwen3_4b_b1_first_eviction_sampled_units():
    w = WORKLOADS["qwen3_4b_b1"]
    units = [(0, 0, 0), (5, 0, 3), (17, 0, 7), (35, 0, 1), (20, 0, 4), (35, 0, 7)]
    rep = run_lockstep(w, seed=0xBEAC1, sample_units=units, steps=w.budget + w.period + 32)
    assert_clean(rep)
    assert rep.units_checked == len(units) * rep.evictions


def test_qwen3_4b_b1_every_unit():
    """The Qwen3-4B single-sequence configuration: its one eviction over all
    36 layers checked on every one of its 288 units (the oracles run in
    parallel worker processes)."""
    w = WORKLOADS["qwen3_4b_b1"]
    rep = run_lockstep_parallel(w, seed=0xBEAC1, steps=w.budget + w.period)
    assert_clean(rep)
    assert rep.evictions == 1 and rep.units_checked == w.units == 288


# Long horizon: each configuration's own stream length on its head shape, with a
# small batch and layer count so that the oracles keep up; every unit checked at
# every eviction (continual FPS across thousands of evictions, ring-slot and
# trace arithmetic at large steps, RoPE angles at positions up to 32K).

def test_long_horizon_r1_qwen7b_32768_steps():
    """R1-Distill-Qwen-7B head shape (GQA 7, theta 1e4, budget 1024): the
    full 32,768-step stream, 1,984 evictions per unit, 8 units."""
    w = WORKLOADS["r1_qwen7b_b128_k1024"].with_(layers=1, batch=2)
    rep = run_lockstep_parallel(w, seed=0xBEAF0, steps=32768)
    assert_clean(rep, min_evictions=1984)
    assert rep.units_checked == 8 * rep.evictions


def test_long_horizon_qwen3_4b_4096_steps():
    """Qwen3-4B head shape (budget 2048): the 4,096-step stream, 128 evictions
    per unit, 2 layers x 2 sequences x 8 KV heads."""
    w = WORKLOADS["qwen3_4b_b192"].with_(layers=2, batch=2)
    rep = run_lockstep_parallel(w, seed=0xBEAF1, steps=4096)
    assert_clean(rep, min_evictions=128)
    assert rep.units_checked == 32 * rep.evictions


def test_long_horizon_qwen3_14b_4096_steps():
    """Qwen3-14B head shape (GQA 5, 8 centres, budget 1024): a 4,096-step
    stream, 192 evictions per unit, 2 sequences x 8 KV heads."""
    w = WORKLOADS["qwen3_14b_b64"].with_(layers=1, batch=2)
    rep = run_lockstep_parallel(w, seed=0xBEAF2, steps=4096)
    assert_clean(rep, min_evictions=192)
    assert rep.units_checked == 16 * rep.evictions


def test_qwen3_4b_b192_full_size_sampled_units():
    """The benchmark workload at full size (58 GB of K/V, 55,296 units, the
    bench's launch configuration), checked on sampled units over three
    evictions, inputs generated on the device."""
    w = WORKLOADS["qwen3_4b_b192"]
    units = [(0, 0, 0), (3, 191, 7), (11, 64, 2), (17, 100, 5), (24, 17, 3), (35, 150, 6),
             (35, 191, 0), (8, 1, 1)]
    rep = run_lockstep(w, seed=0xBEAC2, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period)
    assert_clean(rep, min_evictions=3)
    assert rep.units_checked == len(units) * rep.evictions


def test_qwen3_4b_b192_full_size_without_kept_scores():
    """The bench's own handle configuration (no per-key scores kept) at full
    size: keep sets judged against the oracle's scores, compaction and FPS
    state byte-exact, three evictions on sampled units."""
    w = WORKLOADS["qwen3_4b_b192"]
    units = [(1, 5, 4), (30, 190, 2), (12, 77, 7), (35, 0, 0)]
    rep = run_lockstep(w, seed=0xBEADA, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period, keep_scores=False)
    assert_clean(rep, min_evictions=3)
    assert rep.units_checked == len(units) * rep.evictions


def test_qwen3_14b_b64_full_size_sampled_units():
    """Qwen3-14B head shape (GQA 5, 160 observation rows, budget 1024) at
    batch 64: full-size cache, three evictions, sampled units."""
    w = WORKLOADS["qwen3_14b_b64"]
    units = [(0, 0, 0), (39, 63, 7), (20, 31, 4), (7, 50, 1), (33, 12, 6), (39, 0, 3)]
    rep = run_lockstep(w, seed=0xBEAC3, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period)
    assert_clean(rep, min_evictions=3)
    assert rep.units_checked == len(units) * rep.evictions


@pytest.mark.parametrize("budget", [256, 512, 1024, 2048, 4096])
def test_r1_qwen7b_b128_full_size_sampled_units(budget):
    """R1-Distill-Qwen-7B head shape (GQA 7, 224 observation rows, theta 1e4)
    at batch 128 over every budget of the sweep: full-size cache, three
    evictions, sampled units."""
    w = WORKLOADS[f"r1_qwen7b_b128_k{budget}"]
    units = [(0, 0, 0), (27, 127, 3), (13, 64, 1), (5, 100, 2), (21, 7, 0)]
    rep = run_lockstep(w, seed=0xBEAC4 + budget, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period)
    assert_clean(rep, min_evictions=3)
    assert rep.units_checked == len(units) * rep.evictions


# ---------------------------------------------------------------------------- order-free compaction

@pytest.mark.parametrize("name,over", [
    ("base", dict()),
    ("long_period", dict(period=24)),
    ("no_prefix_no_recent", dict(prefix=0, recent=0)),
    ("gqa7", dict(heads=7, kv_heads=1)),
    ("ragged_budget", dict(budget=200, steps=300)),
    ("batch_layers", dict(layers=2, batch=3, heads=8, kv_heads=2, steps=200)),
])
def test_order_free_tiny_variants(name, over):
    """Order-free compaction over whole tiny streams: the same keep sets as the
    oracle, the holes-from-the-tail layout, byte-exact K/V, and every later
    eviction (which scores the scrambled slots) still matching."""
    w = TINY.with_(**over)
    rep = run_lockstep(w, seed=0xBEAC5, order_free=True)
    assert_clean(rep, min_evictions=3)


def test_order_free_qwen3_4b_b192_full_size_sampled_units():
    w = WORKLOADS["qwen3_4b_b192"]
    units = [(0, 0, 0), (3, 191, 7), (17, 100, 5), (35, 150, 6), (8, 1, 1)]
    rep = run_lockstep(w, seed=0xBEAC6, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period, order_free=True)
    assert_clean(rep, min_evictions=3)
    assert rep.units_checked == len(units) * rep.evictions


def test_order_free_r1_qwen7b_b128_k4096_full_size_sampled_units():
    w = WORKLOADS["r1_qwen7b_b128_k4096"]
    units = [(0, 0, 0), (27, 127, 3), (13, 64, 1)]
    rep = run_lockstep(w, seed=0xBEAC7, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period, order_free=True)
    assert_clean(rep, min_evictions=3)


def test_order_free_needs_recent_window_inside_the_tail():
    from kv_cache_eviction_head_gb300 import bkv
    w = TINY
    dev = torch.device("cuda")
    cfg = bkv.make_config(heads=4, kv_heads=1, d=128, budget=w.budget, period=8, prefix=4,
                          recent=16, layers=1, batch=1, max_cache=w.max_cache, rope_theta=1e6,
                          flags=bkv.BKV_FLAG_ORDER_FREE)
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    q = torch.randn(1, 1, 4, 128, device=dev).to(torch.bfloat16)
    K = [torch.zeros(1, 1, w.max_cache, 128, dtype=torch.bfloat16, device=dev)]
    kept = torch.empty(1, 1, 1, w.budget, dtype=torch.int32, device=dev)
    try:
        for t in range(w.budget + 8):
            bkv.bkv_append_queries(h, q, t)
        with pytest.raises(bkv.BkvError) as e:           # recent 16 > cache_len - budget = 8
            bkv.bkv_evict(h, K, K, w.budget + 8, w.budget + 7, kept)
        assert e.value.code == bkv.BKV_ERR_INVALID_ARG
        for t in range(w.budget + 8, w.budget + 16):
            bkv.bkv_append_queries(h, q, t)
        bkv.bkv_evict(h, K, K, w.budget + 16, w.budget + 15, kept)  # recent 16 <= 16: accepted
        bkv.bkv_sync(h)
    finally:
        bkv.bkv_destroy(h)


# ---------------------------------------------------------------------------- row chunks

@pytest.mark.parametrize("name,over", [
    # G x (16 beacons + 16 recents) observation rows per unit
    ("gqa12_384_rows", dict(heads=12, kv_heads=1)),        # 2 chunks of 192
    ("gqa16_512_rows", dict(heads=16, kv_heads=1)),        # 2 chunks of 256
    ("gqa20_640_rows", dict(heads=20, kv_heads=1)),        # 3 chunks: 214, 214, 212
    ("gqa9_two_kv_288_rows", dict(heads=18, kv_heads=2)),  # 2 chunks of 144
])
@pytest.mark.parametrize("pool", ["max", "mean"])
def test_row_chunks_tiny(name, over, pool):
    """Units with more than 256 observation rows are scored chunk by chunk:
    per-chunk log-sum-exp, then the pooled value carried across chunks."""
    w = TINY.with_(**{"steps": 240, **over})
    rep = run_lockstep(w, seed=0xBEAE0 + len(name), pool=pool)
    assert_clean(rep, min_evictions=3)


def test_row_chunks_order_free_many_tiles():
    w = TINY.with_(heads=12, kv_heads=1, budget=700, steps=800)
    rep = run_lockstep(w, seed=0xBEAE8, order_free=True)
    assert_clean(rep, min_evictions=3)


# ---------------------------------------------------------------------------- the pages' variants

@pytest.mark.parametrize("name,over", [
    ("base", dict()),
    ("gqa7", dict(heads=7, kv_heads=1)),
    ("zero_beacons", dict(fps_cap=16, fps_keep=0)),
    ("ragged_budget", dict(budget=200, steps=300)),
])
def test_mean_pool_tiny_variants(name, over):
    """Mean pooling over queries and heads (Table 2's ablation) on whole tiny
    streams: scores within tolerance, keep sets, compaction and FPS as ever."""
    w = TINY.with_(**over)
    rep = run_lockstep(w, seed=0xBEAC8 + len(name), pool="mean")
    assert_clean(rep, min_evictions=3)


def test_mean_pool_r1_qwen7b_b128_k1024_full_size_sampled_units():
    """Mean pooling at full size on the shape Table 2 uses (R1-Distill-Qwen-7B)."""
    w = WORKLOADS["r1_qwen7b_b128_k1024"]
    units = [(0, 0, 0), (27, 127, 3), (13, 64, 1), (21, 7, 2)]
    rep = run_lockstep(w, seed=0xBEAC9, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + 2 * w.period, pool="mean")
    assert_clean(rep, min_evictions=3)


@pytest.mark.parametrize("recent,beacons", [(4, 28), (1, 31), (31, 1)])
def test_recent_beacon_splits(recent, beacons):
    """Table 1's splits of the 32 observation queries per head: n_rq recent
    queries and fps_keep beacons (4 + 28, 1 + 31, 31 + 1)."""
    w = TINY.with_(fps_cap=32, fps_keep=beacons, steps=400)
    assert w.fps_cap - w.fps_keep == recent
    rep = run_lockstep(w, seed=0xBEACA + recent)
    assert_clean(rep, min_evictions=10)


def test_seven_eighths_schedule_tiny():
    """The pages' schedule at tiny scale: B_max = 256 cut to 7/8 = 224, so 32
    slots drop per eviction and 32 steps separate evictions."""
    w = TINY.with_(budget=224, period=32, steps=600)
    rep = run_lockstep(w, seed=0xBEACB)
    assert_clean(rep, min_evictions=8)


@pytest.mark.parametrize("period", [48, 64])
def test_large_drop_counts_tiny(period):
    """More than 32 drops per eviction take the selector's radix path."""
    w = TINY.with_(budget=160, period=period, steps=520)
    rep = run_lockstep(w, seed=0xBEACD + period)
    assert_clean(rep, min_evictions=5)
    rep = run_lockstep(w, seed=0xBEACD + period, order_free=True)
    assert_clean(rep, min_evictions=5)


def test_seven_eighths_schedule_qwen3_4b_b192_full_size_sampled_units():
    """B_max = 2048 cut to 1792 at full size: 256 drops per unit and eviction,
    FPS every 16 appends between evictions, in slot order and order-free."""
    w = WORKLOADS["qwen3_4b_b192_sched78"]
    units = [(0, 0, 0), (35, 191, 7), (17, 100, 5), (8, 1, 1)]
    for order_free in (False, True):
        rep = run_lockstep(w, seed=0xBEACC, sample_units=units, gen_device="cuda",
                           steps=w.max_cache + w.period, order_free=order_free)
        assert_clean(rep, min_evictions=2)
        assert rep.units_checked == len(units) * rep.evictions


# ---------------------------------------------------------------------------- coverage diagnostic

def test_coverage_tiny_stream():
    """bkv_coverage before every eviction of a whole tiny stream, 40 future
    queries per head (two warps' worth), bit-exact against the oracle."""
    rep = run_lockstep(TINY, seed=0xBEACE, coverage_n=40)
    assert_clean(rep, min_evictions=24)
    assert rep.coverage_checked == 4 * 40 * rep.evictions


def test_coverage_wide_exponents_and_splits():
    """Coverage through the wide-exponent path (future and observation rows
    spanning far more than 20 binades, zero rows, duplicates) and with up to
    62 observation rows per head (31 recents)."""
    w = TINY.with_(steps=300)
    rep = run_lockstep(w, seed=0xBEACF, query_hook=wide_queries, coverage_n=16)
    assert_clean(rep, min_evictions=5)
    w2 = TINY.with_(fps_cap=32, fps_keep=1, steps=300)
    rep = run_lockstep(w2, seed=0xBEAD0, coverage_n=8)
    assert_clean(rep, min_evictions=5)


def test_coverage_qwen3_4b_b192_full_size_sampled_units():
    w = WORKLOADS["qwen3_4b_b192"]
    units = [(0, 0, 0), (35, 191, 7), (17, 100, 5)]
    rep = run_lockstep(w, seed=0xBEAD1, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + w.period, coverage_n=8)
    assert_clean(rep, min_evictions=2)
    assert rep.coverage_checked == len(units) * w.group * 8 * rep.evictions


# ---------------------------------------------------------------------------- prefill

@pytest.mark.parametrize("P", [10, 20, 100, 144])
def test_prefill_tiny(P):
    """Prefill over the stream's first P steps: all recent (P <= n_rq), every
    older query kept (N <= fps_keep), FPS over 84 older queries, and a prompt
    of budget + period evicted at once; the stream then continues in lockstep."""
    w = TINY.with_(steps=320)
    rep = run_lockstep(w, seed=0xBEAD2 + P, prefill=P)
    assert_clean(rep, min_evictions=4)


def test_prefill_long_prompt_then_large_eviction():
    """A 700-step prompt: FPS over 684 older queries per head, then one
    eviction from 700 slots to 128 (572 drops: the radix select) and decoding."""
    w = TINY.with_(cache_slots=700, steps=800)
    rep = run_lockstep(w, seed=0xBEAD3, prefill=700)
    assert_clean(rep, min_evictions=4)


def test_prefill_rows_beyond_shared_memory():
    """A 900-step prompt: 884 older queries per head do not fit the resident
    layout (884 x 272 B), so prefill FPS takes the variant that reads the rows
    from global memory on every pass; queries with wide exponent ranges, zero
    rows and duplicates included."""
    w = TINY.with_(cache_slots=900, steps=960)
    rep = run_lockstep(w, seed=0xBEAD7, prefill=900, query_hook=wide_queries)
    assert_clean(rep, min_evictions=3)


def test_prefill_gqa7_wide_exponents():
    # 96 prompt steps keep the FPS phase of a plain stream: at each eviction a
    # head holds 16 beacons + 16 recents, so 7 heads make 224 observation rows
    w = TINY.with_(heads=7, kv_heads=1, steps=260)
    rep = run_lockstep(w, seed=0xBEAD4, prefill=96, query_hook=wide_queries)
    assert_clean(rep, min_evictions=3)


@pytest.mark.parametrize("pool", ["max", "mean"])
def test_prefill_gqa7_off_phase_266_rows(pool):
    # a prompt of 90 leaves 22 beacons + 16 recents per head at the first
    # evictions: 7 x 38 = 266 observation rows, scored in two chunks of 133
    w = TINY.with_(heads=7, kv_heads=1, steps=260)
    rep = run_lockstep(w, seed=0xBEAD6, prefill=90, pool=pool)
    assert_clean(rep, min_evictions=3)


def test_prefill_qwen3_4b_b192_full_size_sampled_units():
    w = WORKLOADS["qwen3_4b_b192"]
    units = [(0, 0, 0), (35, 191, 7)]
    rep = run_lockstep(w, seed=0xBEAD5, sample_units=units, gen_device="cuda",
                       steps=w.max_cache + w.period, prefill=200)
    assert_clean(rep, min_evictions=2)


def wide_queries(t, q):
    """Replaces some queries by vectors whose exponents span far more than 20
    binades (FPS's wide exact-sum path), by zero rows and by exact duplicates."""
    g = torch.Generator().manual_seed(t)
    out = q.clone()
    if t % 3 == 0:
        e = torch.randint(-60, 8, (q.shape[-1],), generator=g).float()
        s = torch.where(torch.rand(q.shape[-1], generator=g) < 0.5, -1.0, 1.0)
        out[..., 0, :] = (s * (1 + torch.rand(q.shape[-1], generator=g)) * torch.exp2(e)).to(q.dtype)
    if t % 7 == 0:
        out[..., 1, :] = 0
    if t % 5 == 0:
        out[..., 2, :] = out[..., 3, :]
    return out


def test_fps_wide_exponents_zero_rows_duplicates():
    w = TINY.with_(steps=300)
    rep = run_lockstep(w, seed=3, query_hook=wide_queries)
    assert_clean(rep)


EDGE_SCALES = [-42, -41, -40, -39, 18, 19, 20, 21, 90, -110]


def edge_magnitude_queries(t, q):
    """Scales whole query rows by 2^s around the limits of the range FPS uses
    rows as loaded in ([2^-40, 2^21) for the largest component of every
    8-element piece), next to ordinary rows of the same head; one row per
    step gets a piece of nonzero components all below 2^-40."""
    out = q.clone()
    s = EDGE_SCALES[t % len(EDGE_SCALES)]
    out[..., 0, :] = (q[..., 0, :].float() * 2.0 ** s).to(q.dtype)
    out[..., 1, :] = (q[..., 1, :].float() * 2.0 ** EDGE_SCALES[(t // 3) % len(EDGE_SCALES)]).to(q.dtype)
    if t % 4 == 1:
        piece = 8 * (t % 16)
        out[..., 2, piece:piece + 8] = (q[..., 2, piece:piece + 8].float() * 2.0 ** -60).to(q.dtype)
    return out


def test_fps_rows_at_the_raw_range_edges():
    w = TINY.with_(steps=300)
    rep = run_lockstep(w, seed=5, query_hook=edge_magnitude_queries)
    assert_clean(rep)


def test_step_order_and_cache_length_are_validated():
    from kv_cache_eviction_head_gb300 import bkv
    w = TINY
    dev = torch.device("cuda")
    cfg = bkv.make_config(heads=4, kv_heads=1, d=128, budget=w.budget, period=16, prefix=4,
                          recent=16, layers=1, batch=1, max_cache=w.max_cache, rope_theta=1e6)
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    q = torch.randn(1, 1, 4, 128, device=dev).to(torch.bfloat16)
    K = [torch.zeros(1, 1, w.max_cache, 128, dtype=torch.bfloat16, device=dev)]
    kept = torch.empty(1, 1, 1, w.budget, dtype=torch.int32, device=dev)
    try:
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_evict(h, K, K, 5, 0, kept)           # nothing appended yet
        assert e.value.code == bkv.BKV_ERR_STATE
        bkv.bkv_append_queries(h, q, 10)
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_append_queries(h, q, 12)             # skipped a step
        assert e.value.code == bkv.BKV_ERR_STATE
        bad = torch.empty(4 * 128 + 1, dtype=torch.bfloat16, device=dev)
        assert bkv.raw_status("bkv_append_queries", ctypes.c_void_p(h.ptr),
                              ctypes.c_void_p(bad.data_ptr() + 2), 11) == bkv.BKV_ERR_INVALID_ARG
        with pytest.raises(ValueError):                  # the binding checks shapes first
            bkv.bkv_append_queries(h, bad[1:], 11)
        for t in range(11, 11 + w.budget + 15):
            bkv.bkv_append_queries(h, q, t)
        last = 10 + w.budget + 15
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_evict(h, K, K, w.budget + 15, last, kept)  # not the counted length
        assert e.value.code == bkv.BKV_ERR_STATE
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_evict(h, K, K, w.budget + 16, last - 1, kept)  # not the last step
        assert e.value.code == bkv.BKV_ERR_STATE
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_append_queries(h, q, last + 1)         # cache would exceed max_cache
        assert e.value.code == bkv.BKV_ERR_STATE
        bkv.bkv_evict(h, K, K, w.budget + 16, last, kept)
        bkv.bkv_sync(h)
        st = bkv.bkv_get_stats(h)
        assert (st.cache_len, st.beacons, st.recents, st.evictions) == (w.budget, 16, 0, 1)
    finally:
        bkv.bkv_destroy(h)


def test_nonfinite_query_is_latched_not_trapped():
    from kv_cache_eviction_head_gb300 import bkv
    dev = torch.device("cuda")
    cfg = bkv.make_config(heads=4, kv_heads=1, d=128, budget=64, period=16, prefix=4, recent=16,
                          fps_cap=4, fps_keep=2, layers=1, batch=1, max_cache=80, rope_theta=1e6)
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    try:
        for t in range(6):
            q = torch.randn(1, 1, 4, 128, device=dev).to(torch.bfloat16)
            if t == 1:
                q[0, 0, 2, 5] = float("nan")
            bkv.bkv_append_queries(h, q, t)    # the 6th push runs FPS over the NaN row
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_sync(h)
        assert e.value.code == bkv.BKV_ERR_NONFINITE
        bkv.bkv_sync(h)                         # the latch was cleared
    finally:
        bkv.bkv_destroy(h)


def test_bounded_wait_runs_out_latches_timeout_and_the_handle_stays_usable():
    """The bounded device-side waits every kernel uses: four warps wait on a
    barrier nothing completes (about a millisecond here); the wait that runs
    out latches BKV_ERR_TIMEOUT, the other warps see the abort flag and leave,
    and the handle then evicts as usual."""
    from kv_cache_eviction_head_gb300 import bkv
    dev = torch.device("cuda")
    cfg = bkv.make_config(heads=4, kv_heads=1, d=128, budget=64, period=16, prefix=4, recent=16,
                          fps_cap=32, fps_keep=16, layers=1, batch=1, max_cache=80, rope_theta=1e6)
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    try:
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_selftest_wait(h, 0)
        assert e.value.code == bkv.BKV_ERR_INVALID_ARG
        bkv.bkv_selftest_wait(h, 2_000_000)
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_sync(h)
        assert e.value.code == bkv.BKV_ERR_TIMEOUT
        bkv.bkv_sync(h)  # the latch was cleared
        g = torch.Generator(device=dev).manual_seed(3)
        K = [torch.randn(1, 1, 80, 128, generator=g, device=dev).to(torch.bfloat16)]
        V = [torch.randn(1, 1, 80, 128, generator=g, device=dev).to(torch.bfloat16)]
        kept = torch.empty(1, 1, 1, 64, dtype=torch.int32, device=dev)
        for t in range(80):
            bkv.bkv_append_queries(h, torch.randn(1, 1, 4, 128, generator=g, device=dev).to(torch.bfloat16), t)
        bkv.bkv_evict(h, K, V, 80, 79, kept)
        bkv.bkv_sync(h)
        k = kept[0, 0, 0].tolist()
        assert len(k) == 64 and k == sorted(set(k)) and k[:4] == [0, 1, 2, 3] and k[-16:] == list(range(64, 80))
    finally:
        bkv.bkv_destroy(h)
