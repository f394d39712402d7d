"""Device-side error reporting through the C ABI, with inputs made on the host.

A key holding NaN, +inf or -inf must come back from bkv_sync as
BKV_ERR_NONFINITE (latched on the device, nothing trapped), and the same
handle must then evict correctly once the cache holds finite keys again: its
scores and keep set are checked against the CPU oracle started from the
handle's own state. Softmax over every accessible key (BeaconKV reading notes
§2.1 eq. 4) is where a non-finite key enters the scores.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import UnitOracle, select_keep
from synth import to_bits
from tests.lockstep import SCORE_ATOL, SCORE_RTOL, check_keep_set

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_eviction_head_gb300.build import build
    build()


@pytest.mark.parametrize("poison", ["nan", "inf", "-inf"])
@pytest.mark.parametrize("mean", [False, True])
def test_nonfinite_key_is_latched_and_the_handle_recovers(poison, mean):
    from kv_cache_eviction_head_gb300 import bkv
    dev = torch.device("cuda")
    G, budget, period, prefix, recent, L = 4, 64, 16, 4, 16, 80
    cfg = bkv.make_config(heads=G, kv_heads=1, d=128, budget=budget, period=period, prefix=prefix,
                          recent=recent, fps_cap=32, fps_keep=16, layers=1, batch=1, max_cache=L,
                          rope_theta=1e6,
                          flags=bkv.BKV_FLAG_KEEP_SCORES | (bkv.BKV_FLAG_MEAN_POOL if mean else 0))
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    g = torch.Generator().manual_seed(17 + len(poison))
    K = [torch.randn(1, 1, L, 128, generator=g).to(torch.bfloat16).to(dev)]
    V = [torch.randn(1, 1, L, 128, generator=g).to(torch.bfloat16).to(dev)]
    kept = torch.empty(1, 1, 1, budget, dtype=torch.int32, device=dev)
    try:
        for t in range(L):
            bkv.bkv_append_queries(h, torch.randn(1, 1, G, 128, generator=g).to(torch.bfloat16).to(dev), t)
        K[0][0, 0, 37, 5] = float(poison)
        bkv.bkv_evict(h, K, V, L, L - 1, kept)
        with pytest.raises(bkv.BkvError) as e:
            bkv.bkv_sync(h)
        assert e.value.code == bkv.BKV_ERR_NONFINITE
        first = kept[0, 0, 0].tolist()
        assert len(first) == budget and first == sorted(set(first)) and 0 <= first[0] and first[-1] < L

        # finite keys again: every slot rewritten, one more period appended
        K[0].copy_(torch.randn(1, 1, L, 128, generator=g).to(torch.bfloat16))
        V[0].copy_(torch.randn(1, 1, L, 128, generator=g).to(torch.bfloat16))
        for t in range(L, L + period):
            bkv.bkv_append_queries(h, torch.randn(1, 1, G, 128, generator=g).to(torch.bfloat16).to(dev), t)
        st = bkv.bkv_get_stats(h)
        bq_rows, rq_rows = [], []
        for hq in range(G):
            s = bkv.bkv_get_head_state(h, 0, 0, hq)
            bq_rows.append(s[:st.beacons])
            rq_rows.append([s[32 + tau % 16] for tau in range(L, L + period)])
        t = L + period - 1
        k_bits, v_bits = to_bits(K[0][0, 0].cpu()), to_bits(V[0][0, 0].cpu())  # before the compaction
        bkv.bkv_evict(h, K, V, L, t, kept)
        bkv.bkv_sync(h)                                     # clean: the latch was cleared
        uo = UnitOracle(G, 128, 1e6, budget, prefix, recent, 32, 16, pool="mean" if mean else "max")
        pos = first + list(range(L, L + period))
        uo.load_state(bq_rows, rq_rows, list(range(L, L + period)), k_bits, v_bits, pos)
        s_orc, _ = uo.scores(t)
        s_gpu = bkv.bkv_get_scores(h)[0, 0, 0, :L].astype(np.float64)
        assert np.all(np.abs(s_gpu - s_orc) <= SCORE_ATOL + SCORE_RTOL * np.abs(s_orc))
        gk = kept[0, 0, 0].tolist()
        why = check_keep_set(gk, s_orc, select_keep(s_orc, L, prefix, recent, budget), L, prefix,
                             recent, budget)
        assert why is None, why
    finally:
        bkv.bkv_destroy(h)
