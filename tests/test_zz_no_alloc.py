"""bkv_score_select_noalloc: the scoring step for callers that cannot allocate.

Callers that run from a fixed memory arena, or under a runtime that forbids
cudaMalloc once serving has started, cannot hand the library a workspace. This
entry point gives them the eviction's score + keep-set selection with its only
scratch (the RoPE table) in a static device array. The test feeds it the exact
state a handle holds just before two consecutive evictions and checks, through
the C ABI, that its keep sets equal those bkv_evict returns for the same state
(integers, so exactly equal), on two calls in a row that share the scratch.

Cases: several layers, sequences and KV heads; the largest recent-query count
the scratch table holds (32 recents, no beacons); mean pooling. Each call also
hands the entry point a status word, which must read 0 afterwards.

The file name makes pytest collect it last; it also passes alone in a fresh
process (it builds the library itself).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from synth import WORKLOADS, SyntheticStream

pytestmark = pytest.mark.gpu


def snapshot_state(bkv, h, w):
    n_rq = w.fps_cap - w.fps_keep
    bq = np.zeros((w.layers, w.batch, w.heads, w.fps_cap, w.d), dtype=np.uint16)
    rq = np.zeros((w.layers, w.batch, w.heads, n_rq, w.d), dtype=np.uint16)
    for l in range(w.layers):
        for b in range(w.batch):
            for hq in range(w.heads):
                st = bkv.bkv_get_head_state(h, l, b, hq)
                bq[l, b, hq] = st[:w.fps_cap]
                rq[l, b, hq] = st[w.fps_cap:]
    dev = torch.device("cuda")
    as_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return as_dev(bq), as_dev(rq)


@pytest.mark.parametrize("name,over,mean", [
    ("layers_batch_kv_heads", dict(layers=2, batch=3, heads=8, kv_heads=2), False),
    # n_rq = 32 and period 32: every eviction sees 32 recents and no beacons,
    # the largest row count of the static RoPE table
    ("recents_32", dict(fps_cap=32, fps_keep=0, period=32), False),
    ("mean_pool", dict(layers=2, batch=3, heads=8, kv_heads=2), True),
])
def test_noalloc_keep_sets_match_bkv_evict_on_two_calls(name, over, mean):
    from kv_cache_eviction_head_gb300.build import build
    build()
    from kv_cache_eviction_head_gb300 import bkv

    w = WORKLOADS["tiny"].with_(**over)
    dev = torch.device("cuda")
    stream = SyntheticStream(w, seed=99 + len(name), device="cpu")
    K = [torch.zeros(w.batch, w.kv_heads, w.max_cache, w.d, dtype=torch.bfloat16, device=dev)
         for _ in range(w.layers)]
    V = [torch.zeros_like(K[0]) for _ in range(w.layers)]
    kept_ref = torch.full((w.layers, w.batch, w.kv_heads, w.budget), -1, dtype=torch.int32, device=dev)
    kept_na = torch.full_like(kept_ref, -2)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    cfg = bkv.make_config(heads=w.heads, kv_heads=w.kv_heads, d=w.d, budget=w.budget,
                          period=w.period, prefix=w.prefix, recent=w.recent, fps_cap=w.fps_cap,
                          fps_keep=w.fps_keep, layers=w.layers, batch=w.batch,
                          max_cache=w.max_cache, rope_theta=w.theta,
                          flags=bkv.BKV_FLAG_MEAN_POOL if mean else 0)
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    cs = torch.cuda.current_stream()
    h = bkv.bkv_create(cfg, ws, cs)
    calls = 0
    try:
        cache_len = 0
        for t in range(w.max_cache + w.period):
            q = stream.queries().to(dev)
            k, v = stream.keys_values(t)
            for l in range(w.layers):
                K[l][:, :, cache_len] = k[l].to(dev)
                V[l][:, :, cache_len] = v[l].to(dev)
            bkv.bkv_append_queries(h, q, t)
            cache_len += 1
            if cache_len < w.max_cache:
                continue
            st = bkv.bkv_get_stats(h)
            if name == "recents_32":
                assert (st.beacons, st.recents) == (0, 32)
            bq, rq = snapshot_state(bkv, h, w)
            K_before = [x.clone() for x in K]
            bkv.bkv_score_select_noalloc(cfg, bq, rq, st.beacons, st.recents, K_before,
                                         cache_len, t, kept_na, status, cs)
            bkv.bkv_evict(h, K, V, cache_len, t, kept_ref)
            bkv.bkv_sync(h)
            got, want = kept_na.cpu().numpy(), kept_ref.cpu().numpy()
            assert np.array_equal(got, want), f"call {calls + 1}: keep sets differ"
            assert np.all(np.diff(got, axis=-1) > 0)
            assert int(status.item()) == 0, f"call {calls + 1}: device status {int(status.item())}"
            calls += 1
            kept_na.fill_(-2)
            status.fill_(7)
            cache_len = w.budget
    finally:
        bkv.bkv_destroy(h)
    assert calls == 2
