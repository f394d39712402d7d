"""Runs a synthetic decode stream through the CUDA library and the CPU oracle
side by side and compares every eviction.

Agreement rules (per unit and eviction):
  * state before the eviction: every query head's beacons and recent ring equal
    the oracle's, byte for byte (covers every FPS that ran during appends);
  * scores: |s_gpu - s_orc| <= 1e-6 + 2e-3 * |s_orc| for every slot j < L;
  * keep set: exactly `budget` ascending slots, containing the prefix and the
    recent window, and identical to the oracle's on every candidate whose
    oracle score lies farther than 1e-6 + 2e-3 * s_k from s_k, the k_sel-th
    largest candidate score;
  * compaction: K[:budget] and V[:budget] equal the oracle's gather, byte for
    byte, under the keep set the GPU returned once it passed the rule above
    (the oracle continues from that keep set so that an accepted choice inside
    the tie band does not make later rounds diverge);
  * order-free compaction (order_free=True): the returned layout is exactly the
    oracle's order_free_layout of the returned set, and K/V follow it;
  * FPS traces after the eviction: identical pick order for every query head;
  * with coverage_n > 0, before each eviction: bkv_coverage over coverage_n
    seeded future queries equals the oracle's coverage bit for bit (float64);
  * with prefill = P > 0, the stream's first P steps arrive as one prompt
    through bkv_prefill: its picks equal the oracle's prefill FPS trace, and
    when P > budget the prompt is evicted at once (step P - 1, cache P).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from oracle import UnitOracle, order_free_layout, select_keep
from synth import SyntheticStream, Workload, to_bits

SCORE_RTOL = 2e-3
SCORE_ATOL = 1e-6


@dataclass
class LockstepReport:
    evictions: int = 0
    units_checked: int = 0
    kept_adopted: int = 0          # checks where the GPU chose differently inside the tie band
    fps_heads_checked: int = 0
    max_score_rel: float = 0.0
    rows_moved: int = 0
    coverage_checked: int = 0      # (head, future query) values compared
    failures: list = field(default_factory=list)


def check_keep_set(gpu_kept, s_orc, orc_kept, L, prefix, recent, budget):
    """Returns None if the GPU keep set is acceptable, else a reason."""
    g = [int(x) for x in gpu_kept]
    if len(g) != budget or any(b <= a for a, b in zip(g, g[1:])):
        return "keep set not strictly ascending or wrong size"
    gs = set(g)
    if not set(range(prefix)) <= gs or not set(range(L - recent, L)) <= gs:
        return "keep set misses a prefix or recent slot"
    if min(g) < 0 or max(g) >= L:
        return "keep set slot out of range"
    cands = np.arange(prefix, L - recent)
    k_sel = budget - prefix - recent
    s_k = np.sort(s_orc[cands])[::-1][k_sel - 1] if k_sel > 0 else np.inf
    band = SCORE_ATOL + SCORE_RTOL * abs(s_k)
    os_ = set(orc_kept)
    for j in cands:
        if abs(s_orc[j] - s_k) > band and ((j in gs) != (j in os_)):
            return f"slot {j} (score {s_orc[j]:.9g}, k-th {s_k:.9g}) kept differently"
    return None


def run_lockstep(w: Workload, seed: int, sample_units=None, gen_device: str = "cpu",
                 steps: int | None = None, max_failures: int = 20,
                 query_hook=None, order_free: bool = False, pool: str = "max",
                 coverage_n: int = 0, prefill: int = 0) -> LockstepReport:
    from kv_cache_eviction_head_gb300 import bkv

    dev = torch.device("cuda")
    steps = w.steps if steps is None else steps
    G, d = w.group, w.d
    stream = SyntheticStream(w, seed, gen_device)
    K = [torch.zeros(w.batch, w.kv_heads, w.max_cache, d, dtype=torch.bfloat16, device=dev)
         for _ in range(w.layers)]
    V = [torch.zeros_like(K[0]) for _ in range(w.layers)]
    kept = torch.full((w.layers, w.batch, w.kv_heads, w.budget), -1, dtype=torch.int32, device=dev)
    cfg = bkv.make_config(heads=w.heads, kv_heads=w.kv_heads, d=d, budget=w.budget,
                          period=w.period, prefix=w.prefix, recent=w.recent, fps_cap=w.fps_cap,
                          fps_keep=w.fps_keep, layers=w.layers, batch=w.batch,
                          max_cache=w.max_cache, rope_theta=w.theta,
                          flags=bkv.BKV_FLAG_KEEP_SCORES
                          | (bkv.BKV_FLAG_ORDER_FREE if order_free else 0)
                          | (bkv.BKV_FLAG_MEAN_POOL if pool == "mean" else 0))
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())

    if sample_units is None:
        sample_units = [(l, b, kh) for l in range(w.layers) for b in range(w.batch)
                        for kh in range(w.kv_heads)]
    oracles = {u: UnitOracle(G, d, w.theta, w.budget, w.prefix, w.recent, w.fps_cap, w.fps_keep,
                             order_free=order_free, pool=pool)
               for u in sample_units}
    live = set(sample_units)
    idx_dev = torch.device(gen_device)
    l_idx = torch.tensor([u[0] for u in sample_units], device=idx_dev)
    b_idx = torch.tensor([u[1] for u in sample_units], device=idx_dev)
    kh_idx = torch.tensor([u[2] for u in sample_units], device=idx_dev)
    rep = LockstepReport()
    n_rq = w.fps_cap - w.fps_keep

    def fail(msg):
        if len(rep.failures) < max_failures:
            rep.failures.append(msg)

    def evict_and_check(t, cache_len):
        # state before the eviction, byte for byte
        nb_gpu = bkv.bkv_get_stats(h).beacons
        for (l, b, kh) in sorted(live):
            uo = oracles[(l, b, kh)]
            for hg, st in enumerate(uo.heads):
                gst = bkv.bkv_get_head_state(h, l, b, kh * G + hg)
                ok = len(st.bq) == nb_gpu and all(
                    np.array_equal(gst[i], r) for i, r in enumerate(st.bq))
                ok = ok and all(np.array_equal(gst[w.fps_cap + tau % n_rq], r)
                                for r, tau in st.rq)
                if not ok:
                    fail(f"t={t} unit {(l, b, kh)} head {hg}: beacon/recent state differs")
                    live.discard((l, b, kh))
                    break

        if coverage_n > 0:
            g = torch.Generator().manual_seed(seed * 7919 + t)
            qf = (torch.randn(coverage_n, w.layers, w.batch, w.heads, d, generator=g)
                  * torch.exp2(torch.randint(-3, 4, (coverage_n, 1, 1, w.heads, 1), generator=g).float())
                  ).to(torch.bfloat16)
            if query_hook is not None:
                qf = torch.stack([query_hook(t + 1 + i, qf[i]) for i in range(coverage_n)])
            cov = torch.empty(w.layers, w.batch, w.heads, coverage_n, dtype=torch.float64, device=dev)
            bkv.bkv_coverage(h, qf.to(dev), cov)
            cov_h = cov.cpu().numpy()
            qf_bits = to_bits(qf)
            for (l, b, kh) in sorted(live):
                want = oracles[(l, b, kh)].coverage(
                    [qf_bits[:, l, b, kh * G + hg] for hg in range(G)])
                for hg in range(G):
                    got = cov_h[l, b, kh * G + hg].tolist()
                    rep.coverage_checked += coverage_n
                    if got != want[hg]:
                        i = next(i for i in range(coverage_n) if got[i] != want[hg][i])
                        fail(f"t={t} unit {(l, b, kh)} head {hg}: coverage[{i}] "
                             f"gpu {got[i]!r} orc {want[hg][i]!r}")
                        live.discard((l, b, kh))
                        break
        bkv.bkv_evict(h, K, V, cache_len, t, kept)
        bkv.bkv_sync(h)
        rep.evictions += 1
        scores = bkv.bkv_get_scores(h)
        traces = bkv.bkv_get_fps_trace(h)
        kept_h = kept.cpu().numpy()
        L = cache_len
        for (l, b, kh) in sorted(live):
            uo = oracles[(l, b, kh)]
            s_orc, _ = uo.scores(t)
            s_gpu = scores[l, b, kh, :L].astype(np.float64)
            err = np.abs(s_gpu - s_orc)
            tol = SCORE_ATOL + SCORE_RTOL * np.abs(s_orc)
            rel = float(np.max(err / np.maximum(np.abs(s_orc), 1e-30)))
            rep.max_score_rel = max(rep.max_score_rel, rel)
            if np.any(err > tol):
                j = int(np.argmax(err - tol))
                fail(f"t={t} unit {(l, b, kh)}: score[{j}] gpu {s_gpu[j]:.9g} orc {s_orc[j]:.9g}")
                live.discard((l, b, kh))
                continue
            orc_kept = select_keep(s_orc, L, w.prefix, w.recent, w.budget)
            g_layout = kept_h[l, b, kh].tolist()
            g_kept = sorted(g_layout) if order_free else g_layout
            why = check_keep_set(g_kept, s_orc, orc_kept, L, w.prefix, w.recent, w.budget)
            if not why and order_free and g_layout != order_free_layout(g_kept, w.budget):
                why = "order-free layout differs from the holes-from-the-tail rule"
            if why:
                fail(f"t={t} unit {(l, b, kh)}: {why}")
                live.discard((l, b, kh))
                continue
            if g_kept != orc_kept:
                rep.kept_adopted += 1
            res = uo.evict(t, kept_override=g_kept, score=s_orc)
            kg = to_bits(K[l][b, kh, :w.budget])
            vg = to_bits(V[l][b, kh, :w.budget])
            if not (np.array_equal(kg, np.stack(uo.K)) and np.array_equal(vg, np.stack(uo.V))):
                fail(f"t={t} unit {(l, b, kh)}: compacted K/V differ")
                live.discard((l, b, kh))
                continue
            for hg, tr in enumerate(res.traces):
                want = list(tr) + [-1] * (w.fps_keep - len(tr))
                got = traces[l, b, kh * G + hg].tolist()
                rep.fps_heads_checked += 1
                if got != want:
                    fail(f"t={t} unit {(l, b, kh)} head {hg}: FPS trace {got} != {want}")
                    live.discard((l, b, kh))
                    break
            rep.units_checked += 1

    cache_len = 0
    start = 0
    try:
        if prefill > 0:
            # the stream's first `prefill` steps arrive as one prompt
            qs_l = []
            for t in range(prefill):
                q = stream.queries()
                if query_hook is not None:
                    q = query_hook(t, q)
                k, v = stream.keys_values(t)
                kd, vd = k.to(dev), v.to(dev)
                for l in range(w.layers):
                    K[l][:, :, t] = kd[l]
                    V[l][:, :, t] = vd[l]
                qs_l.append(q)
                ks, vs = to_bits(k[l_idx, b_idx, kh_idx]), to_bits(v[l_idx, b_idx, kh_idx])
                for i, u in enumerate(sample_units):
                    oracles[u].append_kv(ks[i], vs[i], t)
            qp = torch.stack(qs_l)                                  # [P][layers][batch][heads][d]
            nr0 = min(n_rq, prefill)
            m0 = min(w.fps_keep, prefill - nr0)
            tr = torch.full((w.layers, w.batch, w.heads, max(m0, 1)), -7, dtype=torch.int32, device=dev)
            bkv.bkv_prefill(h, qp.to(dev), 0, tr if m0 > 0 else None)
            qp_bits = to_bits(qp[:, l_idx, b_idx])                 # [P][units][heads][d]
            tr_h = tr.cpu().numpy()
            for i, (l, b, kh) in enumerate(sample_units):
                uo = oracles[(l, b, kh)]
                uo.prefill([qp_bits[:, i, kh * G + hg] for hg in range(G)], 0)
                for hg, st in enumerate(uo.heads):
                    got = tr_h[l, b, kh * G + hg, :m0].tolist() if m0 > 0 else []
                    rep.fps_heads_checked += 1
                    if got != list(st.trace):
                        fail(f"prefill unit {(l, b, kh)} head {hg}: picks {got} != {list(st.trace)}")
                        live.discard((l, b, kh))
            cache_len = prefill
            start = prefill
            if prefill > w.budget:                                  # evict the prompt down to the budget
                evict_and_check(prefill - 1, cache_len)
                cache_len = w.budget
        for t in range(start, steps):
            q = stream.queries()
            if query_hook is not None:
                q = query_hook(t, q)
            k, v = stream.keys_values(t)
            qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
            for l in range(w.layers):
                K[l][:, :, cache_len] = kd[l]
                V[l][:, :, cache_len] = vd[l]
            bkv.bkv_append_queries(h, qd, t)
            # only the sampled units' rows travel to the host
            qs = to_bits(q[l_idx, b_idx])            # [units][heads][d]
            ks = to_bits(k[l_idx, b_idx, kh_idx])    # [units][d]
            vs = to_bits(v[l_idx, b_idx, kh_idx])
            for i, (l, b, kh) in enumerate(sample_units):
                uo = oracles[(l, b, kh)]
                uo.append_kv(ks[i], vs[i], t)
                uo.append_queries(qs[i, kh * G:(kh + 1) * G], t)
            cache_len += 1
            if cache_len < w.budget + w.period:
                continue

            evict_and_check(t, cache_len)
            cache_len = w.budget
        rep.rows_moved = int(bkv.bkv_get_stats(h).rows_moved)
    finally:
        bkv.bkv_destroy(h)
    return rep
