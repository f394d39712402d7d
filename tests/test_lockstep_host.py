"""Host-side checks of the parity harness (tests/lockstep.py) without a GPU.

The per-unit agreement check and the parallel workers are fed results made by
a second, independent run of the oracle standing in for the library: they must
accept them, and must reject them once a mistake is planted in them (a flipped
K byte, a swapped kept slot, a changed FPS pick, a wrong score)."""

from __future__ import annotations

import queue

import numpy as np
import pytest
import torch

from oracle import UnitOracle, select_keep
from synth import WORKLOADS, SyntheticStream, to_bits
from tests.lockstep import GpuUnitResult, LockstepReport, _unit_worker, check_unit

W = WORKLOADS["tiny"].with_(layers=1, batch=2, heads=8, kv_heads=2, steps=200)


def library_stand_in(w, seed, units, plant=None):
    """Runs the stream through reference oracles and yields, per eviction,
    (t, L, {unit: GpuUnitResult}) as the library would report them."""
    G, n_rq = w.group, w.fps_cap - w.fps_keep
    stream = SyntheticStream(w, seed, "cpu")
    ref = {u: UnitOracle(G, w.d, w.theta, w.budget, w.prefix, w.recent, w.fps_cap, w.fps_keep) for u in units}
    cache_len = 0
    out = []
    for t in range(w.steps):
        q = stream.queries()
        k, v = stream.keys_values(t)
        qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
        for (l, b, kh), uo in ref.items():
            uo.append_kv(kb[l, b, kh], vb[l, b, kh], t)
            uo.append_queries(qb[l, b, kh * G:(kh + 1) * G], t)
        cache_len += 1
        if cache_len < w.budget + w.period:
            continue
        res = {}
        for u, uo in ref.items():
            nb = len(uo.heads[0].bq)
            state = []
            for st in uo.heads:
                a = np.zeros((w.fps_cap + n_rq, w.d), dtype=np.uint16)
                for i, r in enumerate(st.bq):
                    a[i] = r
                for r, tau in st.rq:
                    a[w.fps_cap + tau % n_rq] = r
                state.append(a)
            s, _ = uo.scores(t)
            ev = uo.evict(t, score=s)
            res[u] = GpuUnitResult(nb=nb, state=state, scores=s.astype(np.float32), layout=list(ev.kept),
                                   K=np.stack(uo.K), V=np.stack(uo.V),
                                   traces=[list(tr) + [-1] * (w.fps_keep - len(tr)) for tr in ev.traces])
        if plant is not None:
            plant(len(out), res)
        out.append((t, cache_len, res))
        cache_len = w.budget
    return out


UNITS = [(0, 0, 0), (0, 1, 1), (0, 0, 1)]


def run_worker(evictions):
    inq, outq = queue.Queue(), queue.Queue()
    for m in evictions:
        inq.put(m)
    inq.put(None)
    _unit_worker(W, 11, UNITS, False, "max", inq, outq)
    return outq.get()


def test_worker_accepts_an_independent_oracle_run():
    ev = library_stand_in(W, 11, UNITS)
    rep = run_worker(ev)
    assert not rep.failures, rep.failures
    assert rep.evictions == len(ev) >= 4
    assert rep.units_checked == len(UNITS) * len(ev)


def _flip_k(i, res):
    if i == 2:
        res[(0, 1, 1)].K[5, 7] ^= 1


def _swap_kept(i, res):
    if i == 1:
        r = res[(0, 0, 0)]
        dropped = sorted(set(range(W.prefix, W.budget + W.period - W.recent)) - set(r.layout))
        r.layout = sorted(set(r.layout) - {r.layout[W.prefix + 3]} | {dropped[0]})


def _change_trace(i, res):
    if i == 3:
        tr = res[(0, 0, 1)].traces[2]
        tr[4], tr[5] = tr[5], tr[4]


def _wrong_score(i, res):
    if i == 0:
        res[(0, 1, 1)].scores[20] *= 1.01


@pytest.mark.parametrize("plant", [_flip_k, _swap_kept, _change_trace, _wrong_score])
def test_worker_rejects_a_planted_mistake(plant):
    rep = run_worker(library_stand_in(W, 11, UNITS, plant=plant))
    assert rep.failures, f"{plant.__name__} went unnoticed"


def test_check_unit_adopts_a_tie_band_choice():
    """Two candidates with equal scores at the k-th place: either keep set is
    accepted, and the oracle continues from the library's choice."""
    w = W.with_(heads=1, kv_heads=1, fps_cap=2, fps_keep=1, budget=8, period=2, prefix=1, recent=1)
    uo = UnitOracle(1, w.d, w.theta, w.budget, w.prefix, w.recent, w.fps_cap, w.fps_keep)
    row = np.zeros(w.d, dtype=np.uint16)
    for t in range(10):
        uo.append_kv(row, row, t)          # all-zero keys: every score ties
        uo.append_queries([row], t)
    s, _ = uo.scores(9)
    want = select_keep(s, 10, w.prefix, w.recent, w.budget)
    dropped = sorted(set(range(1, 9)) - set(want))
    other = sorted(set(want) - {want[-2]} | {dropped[0]})
    assert len(other) == w.budget and other != want
    rep = LockstepReport()
    res = GpuUnitResult(nb=1, state=[np.zeros((3, w.d), dtype=np.uint16)], scores=s.astype(np.float32),
                        layout=other, K=np.zeros((8, w.d), np.uint16), V=np.zeros((8, w.d), np.uint16),
                        traces=[[0]])
    res.state[0][w.fps_cap + 9 % 1] = row
    ok = check_unit(uo, (0, 0, 0), 9, 10, w, res, False, rep, rep.failures.append)
    assert ok, rep.failures
    assert rep.kept_adopted == 1
    assert uo.pos == other


def _drop_scores(i, res):
    for r in res.values():
        r.scores = None


@pytest.mark.parametrize("plant", [None, _flip_k, _swap_kept, _change_trace])
def test_worker_without_kept_scores(plant):
    """With no scores kept (the handle as the throughput run configures it)
    the keep set, the compaction and the FPS state are still compared: a
    correct run passes and each planted mistake is still caught."""
    def both(i, res):
        if plant is not None:
            plant(i, res)
        _drop_scores(i, res)
    rep = run_worker(library_stand_in(W, 11, UNITS, plant=both))
    if plant is None:
        assert not rep.failures, rep.failures
        assert rep.units_checked == len(UNITS) * rep.evictions
    else:
        assert rep.failures, f"{plant.__name__} went unnoticed without scores"
