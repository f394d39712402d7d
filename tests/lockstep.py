"""Runs a synthetic decode stream through the CUDA library and the CPU oracle
side by side and compares every eviction.

Agreement rules (per unit and eviction):
  * state before the eviction: every query head's beacons and recent ring equal
    the oracle's, byte for byte (covers every FPS that ran during appends);
  * scores: |s_gpu - s_orc| <= 1e-6 + 2e-3 * |s_orc| for every slot j < L
    (with keep_scores=False the handle keeps no scores, as in the bench, and
    only the keep set, the compaction and the FPS state are compared, the
    keep set still against the oracle's scores);
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
    evictions_by_unit: dict = field(default_factory=dict)  # unit -> evictions checked


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


@dataclass
class GpuUnitResult:
    """One unit's library outputs at one eviction, copied to the host."""
    nb: int                # beacons per query head before the eviction
    state: list            # per query head: uint16 [fps_cap + n_rq][d] before the eviction
    scores: np.ndarray     # float32 [L], or None when the handle keeps no scores
    layout: list           # kept slots (ascending), or the order-free layout
    K: np.ndarray          # uint16 [budget][d] after the compaction
    V: np.ndarray
    traces: list           # per query head: FPS pick order after the eviction


def check_unit(uo, unit, t, L, w, res: GpuUnitResult, order_free, rep, fail) -> bool:
    """Compares one unit's library outputs at the eviction of step t with its
    oracle and advances the oracle through that eviction (adopting the
    library's keep set once it passed). Returns False at the first mismatch."""
    n_rq = w.fps_cap - w.fps_keep
    for hg, st in enumerate(uo.heads):
        gst = res.state[hg]
        ok = len(st.bq) == res.nb and all(np.array_equal(gst[i], r) for i, r in enumerate(st.bq))
        ok = ok and all(np.array_equal(gst[w.fps_cap + tau % n_rq], r) for r, tau in st.rq)
        if not ok:
            fail(f"t={t} unit {unit} head {hg}: beacon/recent state differs")
            return False
    s_orc, _ = uo.scores(t)
    if res.scores is not None:
        s_gpu = np.asarray(res.scores, dtype=np.float64)
        err = np.abs(s_gpu - s_orc)
        tol = SCORE_ATOL + SCORE_RTOL * np.abs(s_orc)
        rel = float(np.max(err / np.maximum(np.abs(s_orc), 1e-30)))
        rep.max_score_rel = max(rep.max_score_rel, rel)
        if np.any(err > tol):
            j = int(np.argmax(err - tol))
            fail(f"t={t} unit {unit}: score[{j}] gpu {s_gpu[j]:.9g} orc {s_orc[j]:.9g}")
            return False
    orc_kept = select_keep(s_orc, L, w.prefix, w.recent, w.budget)
    g_layout = [int(x) for x in res.layout]
    g_kept = sorted(g_layout) if order_free else g_layout
    why = check_keep_set(g_kept, s_orc, orc_kept, L, w.prefix, w.recent, w.budget)
    if not why and order_free and g_layout != order_free_layout(g_kept, w.budget):
        why = "order-free layout differs from the holes-from-the-tail rule"
    if why:
        fail(f"t={t} unit {unit}: {why}")
        return False
    if g_kept != orc_kept:
        rep.kept_adopted += 1
    ev = uo.evict(t, kept_override=g_kept, score=s_orc)
    if not (np.array_equal(res.K, np.stack(uo.K)) and np.array_equal(res.V, np.stack(uo.V))):
        fail(f"t={t} unit {unit}: compacted K/V differ")
        return False
    for hg, tr in enumerate(ev.traces):
        want = list(tr) + [-1] * (w.fps_keep - len(tr))
        rep.fps_heads_checked += 1
        if list(res.traces[hg]) != want:
            fail(f"t={t} unit {unit} head {hg}: FPS trace {list(res.traces[hg])} != {want}")
            return False
    rep.units_checked += 1
    rep.evictions_by_unit[unit] = rep.evictions_by_unit.get(unit, 0) + 1
    return True


def run_lockstep(w: Workload, seed: int, sample_units=None, gen_device: str = "cpu",
                 steps: int | None = None, max_failures: int = 20,
                 query_hook=None, order_free: bool = False, pool: str = "max",
                 coverage_n: int = 0, prefill: int = 0, keep_scores: bool = True) -> LockstepReport:
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
                          flags=(bkv.BKV_FLAG_KEEP_SCORES if keep_scores else 0)
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
        # state before the eviction, byte for byte (compared in check_unit)
        nb_gpu = bkv.bkv_get_stats(h).beacons
        states = {u: [bkv.bkv_get_head_state(h, u[0], u[1], u[2] * G + hg) for hg in range(G)]
                  for u in sorted(live)}

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
        scores = bkv.bkv_get_scores(h) if keep_scores else None
        traces = bkv.bkv_get_fps_trace(h)
        kept_h = kept.cpu().numpy()
        for (l, b, kh) in sorted(live):
            u = (l, b, kh)
            res = GpuUnitResult(nb=nb_gpu, state=states[u],
                                scores=scores[l, b, kh, :cache_len] if keep_scores else None,
                                layout=kept_h[l, b, kh].tolist(),
                                K=to_bits(K[l][b, kh, :w.budget]), V=to_bits(V[l][b, kh, :w.budget]),
                                traces=[traces[l, b, kh * G + hg].tolist() for hg in range(G)])
            if not check_unit(oracles[u], u, t, cache_len, w, res, order_free, rep, fail):
                live.discard(u)

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


# ---------------------------------------------------------------------------- many units in parallel

def _unit_worker(w: Workload, seed: int, units: list, order_free: bool, pool: str, inq, outq) -> None:
    """Child process: regenerates the seeded stream on the CPU (the same draws
    the parent hands the library), keeps the oracles of `units`, and checks
    every eviction the parent sends, (t, L, {unit: GpuUnitResult}), until None."""
    torch.set_num_threads(1)
    G = w.group
    stream = SyntheticStream(w, seed, "cpu")
    oracles = {u: UnitOracle(G, w.d, w.theta, w.budget, w.prefix, w.recent, w.fps_cap, w.fps_keep,
                             order_free=order_free, pool=pool) for u in units}
    live = set(units)
    rep = LockstepReport()

    def fail(msg):
        if len(rep.failures) < 20:
            rep.failures.append(msg)

    l_idx = torch.tensor([u[0] for u in units])
    b_idx = torch.tensor([u[1] for u in units])
    kh_idx = torch.tensor([u[2] for u in units])
    t_next = 0
    try:
        while True:
            msg = inq.get()
            if msg is None:
                break
            t, L, results = msg
            while t_next <= t:
                q = stream.queries()
                k, v = stream.keys_values(t_next)
                qs = to_bits(q[l_idx, b_idx])
                ks, vs = to_bits(k[l_idx, b_idx, kh_idx]), to_bits(v[l_idx, b_idx, kh_idx])
                for i, (l, b, kh) in enumerate(units):
                    uo = oracles[(l, b, kh)]
                    uo.append_kv(ks[i], vs[i], t_next)
                    uo.append_queries(qs[i, kh * G:(kh + 1) * G], t_next)
                t_next += 1
            rep.evictions += 1
            for u in sorted(live):
                if u not in results or not check_unit(oracles[u], u, t, L, w, results[u], order_free, rep, fail):
                    if u not in results:
                        fail(f"t={t} unit {u}: no library result")
                    live.discard(u)
    except Exception as e:  # reported to the parent as a failure
        fail(f"worker for {units[:3]}...: {type(e).__name__}: {e}")
    outq.put(rep)


def run_lockstep_parallel(w: Workload, seed: int, sample_units=None, steps: int | None = None,
                          workers: int | None = None, order_free: bool = False,
                          pool: str = "max", keep_scores: bool = True) -> LockstepReport:
    """run_lockstep's agreement rules on many units at once: the library runs
    the stream (generated on the CPU) in this process, and the oracles of the
    sampled units run in `workers` spawned child processes that regenerate the
    same stream and check each eviction as it arrives (bounded queues: the
    library waits when the oracles fall behind). No prefill, coverage or
    query hook."""
    import multiprocessing as mp
    import os
    from kv_cache_eviction_head_gb300 import bkv

    dev = torch.device("cuda")
    steps = w.steps if steps is None else steps
    G, d = w.group, w.d
    if sample_units is None:
        sample_units = [(l, b, kh) for l in range(w.layers) for b in range(w.batch)
                        for kh in range(w.kv_heads)]
    n = max(1, min(workers or max(1, len(os.sched_getaffinity(0)) - 1), len(sample_units)))
    groups = [sample_units[i::n] for i in range(n)]
    owner = {u: i for i, grp in enumerate(groups) for u in grp}
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    inqs = [ctx.Queue(maxsize=4) for _ in groups]
    outq = ctx.Queue()
    procs = [ctx.Process(target=_unit_worker, args=(w, seed, grp, order_free, pool, iq, outq), daemon=True)
             for grp, iq in zip(groups, inqs)]
    for p in procs:
        p.start()
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v

    def send(i, msg):
        while True:
            try:
                inqs[i].put(msg, timeout=5)
                return
            except Exception:
                if not procs[i].is_alive():
                    raise RuntimeError(f"oracle worker {i} exited with code {procs[i].exitcode}")

    stream = SyntheticStream(w, seed, "cpu")
    K = [torch.zeros(w.batch, w.kv_heads, w.max_cache, d, dtype=torch.bfloat16, device=dev)
         for _ in range(w.layers)]
    V = [torch.zeros_like(K[0]) for _ in range(w.layers)]
    kept = torch.full((w.layers, w.batch, w.kv_heads, w.budget), -1, dtype=torch.int32, device=dev)
    cfg = bkv.make_config(heads=w.heads, kv_heads=w.kv_heads, d=d, budget=w.budget,
                          period=w.period, prefix=w.prefix, recent=w.recent, fps_cap=w.fps_cap,
                          fps_keep=w.fps_keep, layers=w.layers, batch=w.batch,
                          max_cache=w.max_cache, rope_theta=w.theta,
                          flags=(bkv.BKV_FLAG_KEEP_SCORES if keep_scores else 0)
                          | (bkv.BKV_FLAG_ORDER_FREE if order_free else 0)
                          | (bkv.BKV_FLAG_MEAN_POOL if pool == "mean" else 0))
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = bkv.bkv_create(cfg, ws, torch.cuda.current_stream())
    layers = sorted({u[0] for u in sample_units})
    main = LockstepReport()
    try:
        cache_len = 0
        for t in range(steps):
            q = stream.queries()
            k, v = stream.keys_values(t)
            kd, vd = k.to(dev), v.to(dev)
            for l in range(w.layers):
                K[l][:, :, cache_len] = kd[l]
                V[l][:, :, cache_len] = vd[l]
            bkv.bkv_append_queries(h, q.to(dev), t)
            cache_len += 1
            if cache_len < w.budget + w.period:
                continue
            nb = bkv.bkv_get_stats(h).beacons
            states = {u: [bkv.bkv_get_head_state(h, u[0], u[1], u[2] * G + hg) for hg in range(G)]
                      for u in sample_units}
            bkv.bkv_evict(h, K, V, cache_len, t, kept)
            bkv.bkv_sync(h)
            main.evictions += 1
            scores = bkv.bkv_get_scores(h) if keep_scores else None
            traces = bkv.bkv_get_fps_trace(h)
            kept_h = kept.cpu().numpy()
            kv_h = {l: (to_bits(K[l][:, :, :w.budget]), to_bits(V[l][:, :, :w.budget])) for l in layers}
            msgs = [dict() for _ in groups]
            for u in sample_units:
                l, b, kh = u
                msgs[owner[u]][u] = GpuUnitResult(
                    nb=nb, state=states[u], scores=scores[l, b, kh, :cache_len].copy() if keep_scores else None,
                    layout=kept_h[l, b, kh].tolist(), K=kv_h[l][0][b, kh].copy(), V=kv_h[l][1][b, kh].copy(),
                    traces=[traces[l, b, kh * G + hg].tolist() for hg in range(G)])
            for i, m in enumerate(msgs):
                send(i, (t, cache_len, m))
            cache_len = w.budget
        main.rows_moved = int(bkv.bkv_get_stats(h).rows_moved)
    finally:
        bkv.bkv_destroy(h)
        for i in range(len(groups)):
            try:
                send(i, None)
            except RuntimeError as e:
                main.failures.append(str(e))
    got = 0
    while got < len(groups):
        try:
            r = outq.get(timeout=30)
        except Exception:
            if all(not p.is_alive() for p in procs):
                main.failures.append("an oracle worker exited without a report")
                break
            continue
        got += 1
        main.units_checked += r.units_checked
        main.kept_adopted += r.kept_adopted
        main.fps_heads_checked += r.fps_heads_checked
        main.max_score_rel = max(main.max_score_rel, r.max_score_rel)
        main.failures += r.failures
        main.evictions_by_unit.update(r.evictions_by_unit)
    for p in procs:
        p.join(timeout=30)
    return main
