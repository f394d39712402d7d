"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a closed form, exact rational
arithmetic, an independently written brute force, a textbook identity or a
hand-derived fixture under tests/golden/. None of these call the CUDA path.
"""

from __future__ import annotations

import functools
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import (UnitOracle, attention_weights, bf16_to_f64, cosine_matrix, coverage, exact_dot, fps,
                    gram_exact, max_pool, mean_pool, order_free_layout, rope, select_keep)
from synth import kv_bytes_per_token, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def bf16_bits(x) -> np.ndarray:
    return to_bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def rand_bits(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return to_bits((torch.randn(*shape, generator=g) * scale).to(torch.bfloat16))


# ---------------------------------------------------------------------------- values

def test_bf16_decode_known_patterns():
    assert bf16_to_f64(np.uint16(0x3F80)) == 1.0
    assert bf16_to_f64(np.uint16(0xC000)) == -2.0
    assert bf16_to_f64(np.uint16(0x0001)) == 2.0 ** -133            # smallest subnormal
    assert bf16_to_f64(np.uint16(0x0080)) == 2.0 ** -126            # smallest normal
    assert bf16_to_f64(np.uint16(0x7F7F)) == (2 - 2 ** -7) * 2.0 ** 127
    assert bf16_to_f64(np.uint16(0x3FC0)) == 1.5


# ---------------------------------------------------------------------------- exact Gram

def frac_dot(a_bits, b_bits) -> float:
    fa = [Fraction(float(x)) for x in bf16_to_f64(a_bits)]
    fb = [Fraction(float(x)) for x in bf16_to_f64(b_bits)]
    return float(sum((x * y for x, y in zip(fa, fb)), Fraction(0)))  # correctly rounded


def crafted_vectors():
    """Vectors that break naive fp64 summation: cancellation, subnormals, wide spread."""
    d = 128
    vs = []
    v = np.zeros(d, np.float32); v[0], v[1], v[2] = 2.0 ** 100, 1.0, -(2.0 ** 100); vs.append(v)
    v = np.zeros(d, np.float32); v[:] = 1.0; v[5] = 2.0 ** 60; v[9] = -(2.0 ** 60); vs.append(v)
    v = np.zeros(d, np.float32); v[::2] = 2.0 ** -130; v[1::2] = 3.0 * 2.0 ** -128; vs.append(v)
    v = np.zeros(d, np.float32); v[3] = 2.0 ** 120; v[4] = 2.0 ** -120; v[7] = 1.0 + 2 ** -7; vs.append(v)
    g = np.random.default_rng(7)
    for _ in range(6):
        e = g.integers(-125, 120, size=d)
        v = (g.choice([-1.0, 1.0], size=d) * (1 + g.integers(0, 128, size=d) / 128.0) * 2.0 ** e)
        vs.append(v.astype(np.float32))
    return [bf16_bits(v) for v in vs]


def test_exact_dot_matches_rational_arithmetic():
    vs = crafted_vectors()
    for a, b in itertools.product(vs, vs):
        assert exact_dot(bf16_to_f64(a), bf16_to_f64(b)) == frac_dot(a, b)
    # a case where left-to-right float64 summation is wrong
    a = vs[0]
    ones = bf16_bits(np.ones(128))
    naive = 0.0
    for x in bf16_to_f64(a):
        naive += x
    assert naive == 0.0 and exact_dot(bf16_to_f64(a), bf16_to_f64(ones)) == 1.0


def test_exact_dot_random_rows_match_rational():
    X = rand_bits((12, 128), seed=3, scale=0.1)
    G = gram_exact(bf16_to_f64(X))
    for i in range(12):
        for j in range(12):
            assert G[i][j] == frac_dot(X[i], X[j])


def test_cosine_closed_forms():
    E = np.eye(4, 128)
    C = cosine_matrix(gram_exact(E))
    assert C == [[1.0 if i == j else 0.0 for j in range(4)] for i in range(4)]
    # zero vector convention and Cauchy-Schwarz
    X = np.zeros((3, 128)); X[0, 0] = 3.0; X[0, 1] = 4.0; X[2, 0] = -6.0
    C = cosine_matrix(gram_exact(X))
    assert C[1] == [0.0, 0.0, 0.0] and C[0][1] == 0.0
    assert C[0][2] == -18.0 / math.sqrt(25.0 * 36.0) == -0.6
    Y = bf16_to_f64(rand_bits((20, 128), seed=5))
    for row in cosine_matrix(gram_exact(Y)):
        assert all(abs(c) <= 1.0 + 4e-16 for c in row)


# ---------------------------------------------------------------------------- FPS

def fps_brute(Xbits, m):
    """Independent re-derivation of the greedy rule: every step recomputes each
    candidate's largest cosine to the selected set from scratch; the Gram comes
    from exact rational arithmetic."""
    n = len(Xbits)
    if n <= m:
        return list(range(n))
    if m == 0:
        return []
    G = [[frac_dot(Xbits[i], Xbits[j]) for j in range(n)] for i in range(n)]

    def cos(i, j):
        if G[i][i] == 0.0 or G[j][j] == 0.0:
            return 0.0
        return G[i][j] / math.sqrt(G[i][i] * G[j][j])

    means = [functools.reduce(lambda acc, j: acc + cos(i, j), range(n), 0.0) / n for i in range(n)]
    chosen = [min(range(n), key=lambda i: (means[i], i))]
    while len(chosen) < m:
        rest = [j for j in range(n) if j not in chosen]
        nearest = {j: max(cos(j, r) for r in chosen) for j in rest}
        chosen.append(min(rest, key=lambda j: (nearest[j], j)))
    return chosen


@pytest.mark.parametrize("seed", range(40))
def test_fps_matches_brute_force(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(2, 13))
    m = int(g.integers(1, n + 1))
    X = rand_bits((n, 128), seed=1000 + seed, scale=0.1)
    if seed % 4 == 0:                       # exact duplicates -> exact ties
        X[n // 2] = X[0]
    if seed % 5 == 0:                       # a zero row -> cosine-0 convention
        X[-1] = 0
    if seed % 3 == 0:                       # a few rows from a small shared set -> near ties
        X[1:3] = rand_bits((1, 128), seed=seed)[0]
    trace, kept = fps(bf16_to_f64(X), m)
    assert trace == fps_brute(X, m)
    assert kept == sorted(trace)


def test_fps_golden_axes():
    gd = read_golden("fps_axes.txt")
    vecs = [[float(x) for x in v.split(",")] for v in gd["vectors"].split(";")]
    X = np.zeros((len(vecs), 128))
    for i, v in enumerate(vecs):
        X[i, :len(v)] = v
    Xb = bf16_to_f64(bf16_bits(X))
    trace, kept = fps(Xb, int(gd["m"]))
    assert trace == [int(x) for x in gd["trace"].split(",")]
    assert kept == [int(x) for x in gd["kept"].split(",")]
    # m >= N keeps every row in order: no sampling happens
    assert fps(Xb, len(vecs)) == (list(range(len(vecs))), list(range(len(vecs))))


def test_fps_orthonormal_all_ties_is_index_order():
    X = np.eye(10, 128)
    assert fps(X, 7)[0] == list(range(7))


def test_fps_circle_picks_opposite_points():
    # points on a circle at known angles: start at the least-central point, then
    # the farthest from it, ...
    ang = np.deg2rad([0, 10, 20, 30, 100, 200, 250])
    X = np.zeros((len(ang), 128))
    X[:, 0], X[:, 1] = np.cos(ang), np.sin(ang)
    Xb = bf16_to_f64(bf16_bits(X))
    trace, _ = fps(Xb, 3)
    assert trace == fps_brute(bf16_bits(X), 3)
    C = cosine_matrix(gram_exact(Xb))
    means = [sum(r) / len(r) for r in C]
    assert trace[0] == int(np.argmin(means))
    # the second pick is the point with the lowest cosine to the first
    assert trace[1] == int(np.argmin([C[j][trace[0]] for j in range(len(ang))]))


@pytest.mark.parametrize("seed", range(10))
def test_fps_pick_values_are_nondecreasing(seed):
    X = bf16_to_f64(rand_bits((32, 128), seed=2000 + seed, scale=0.1))
    trace, _ = fps(X, 16)
    C = cosine_matrix(gram_exact(X))
    vals = [max(C[trace[k]][r] for r in trace[:k]) for k in range(1, 16)]
    assert all(b >= a for a, b in zip(vals, vals[1:]))


@pytest.mark.parametrize("seed", range(12))
def test_fps_k_center_two_approximation(seed):
    """Farthest-first traversal covers within twice the optimal angular radius."""
    n, m = 9, 3
    X = bf16_to_f64(rand_bits((n, 128), seed=3000 + seed, scale=0.1))
    C = cosine_matrix(gram_exact(X))
    ang = [[math.acos(max(-1.0, min(1.0, c))) for c in row] for row in C]

    def radius(S):
        return max(min(ang[j][s] for s in S) for j in range(n))

    opt = min(radius(S) for S in itertools.combinations(range(n), m))
    assert radius(fps(X, m)[0]) <= 2 * opt + 1e-12


# ---------------------------------------------------------------------------- RoPE

def test_rope_two_dims_is_plane_rotation():
    x = np.array([0.3, -1.7])
    for pos in (0, 1, 5, 1234):
        c, s = math.cos(pos), math.sin(pos)
        assert np.allclose(rope(x, pos, 1e4), [x[0] * c - x[1] * s, x[1] * c + x[0] * s],
                           rtol=0, atol=1e-14)


def test_rope_four_dims_block_rotation():
    theta, pos = 100.0, 7
    x = np.array([1.0, 2.0, 3.0, 4.0])
    f = [1.0, theta ** -0.5]                  # theta^(-2i/d), i = 0, 1, d = 4
    want = np.empty(4)
    for i in range(2):
        a = pos * f[i]
        want[i] = x[i] * math.cos(a) - x[i + 2] * math.sin(a)
        want[i + 2] = x[i + 2] * math.cos(a) + x[i] * math.sin(a)
    assert np.allclose(rope(x, pos, theta), want, rtol=0, atol=1e-14)


def test_rope_norm_relative_and_identity():
    g = np.random.default_rng(0)
    q, k = g.standard_normal(128), g.standard_normal(128)
    for theta in (1e4, 1e6):
        assert np.allclose(rope(q, 0, theta), q, rtol=0, atol=0)
        for p in (3, 2063, 32767):
            assert abs(np.linalg.norm(rope(q, p, theta)) - np.linalg.norm(q)) < 1e-12
        base = rope(q, 40, theta) @ rope(k, 10, theta)
        for shift in (1, 500, 20000):
            assert abs(rope(q, 40 + shift, theta) @ rope(k, 10 + shift, theta) - base) < 1e-10


# ---------------------------------------------------------------------------- scores

def test_softmax_rows_sum_to_one_and_respect_access():
    g = np.random.default_rng(1)
    Q, K = g.standard_normal((12, 128)), g.standard_normal((50, 128))
    qpos = np.array([49] * 6 + list(range(44, 50)))
    W = attention_weights(Q, qpos, K, np.arange(50))
    assert np.allclose(W.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    for r in range(12):
        assert np.all(W[r, np.arange(50) > qpos[r]] == 0.0)
        assert np.all(W[r, np.arange(50) <= qpos[r]] > 0.0)


def test_single_row_score_is_that_rows_softmax():
    g = np.random.default_rng(2)
    q, K = g.standard_normal(128), g.standard_normal((30, 128))
    logits = [float(q @ K[j]) / math.sqrt(128) for j in range(30)]
    z = sum(math.exp(x) for x in logits)
    want = [math.exp(x) / z for x in logits]
    got = max_pool(attention_weights(q[None, :], [29], K, np.arange(30)))
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def snapkv_max_score(heads_recent, K_vals, k_pos, theta, d):
    """SnapKV-style recent-window max score (eqs. 4-5 of the notes), extra max
    over the query heads of the group, written as explicit loops."""
    L = len(K_vals)
    best = [0.0] * L
    for recent in heads_recent:
        for q, tau in recent:
            qr = rope(bf16_to_f64(q), tau, theta)
            acc = [j for j in range(L) if k_pos[j] <= tau]
            logit = {j: float(qr @ K_vals[j]) / math.sqrt(d) for j in acc}
            mx = max(logit.values())
            z = math.fsum(math.exp(v - mx) for v in logit.values())
            for j in acc:
                best[j] = max(best[j], math.exp(logit[j] - mx) / z)
    return np.array(best)


def test_zero_beacons_reduce_to_snapkv_max_formula():
    G, d = 2, 128
    u = UnitOracle(group=G, d=d, theta=1e6, budget=40, prefix=4, recent=8, fps_cap=16,
                   fps_keep=0)
    g = torch.Generator().manual_seed(11)
    t = 0
    for rnd in range(2):
        while len(u.K) < 56:
            u.append_kv(to_bits(torch.randn(d, generator=g).to(torch.bfloat16)),
                        to_bits(torch.randn(d, generator=g).to(torch.bfloat16)), t)
            u.append_queries(to_bits(torch.randn(G, d, generator=g).to(torch.bfloat16)), t)
            t += 1
        if rnd == 1:                               # after one eviction: no beacons left
            assert all(len(st.bq) == 0 for st in u.heads)
            got, nobs = u.scores(t - 1)
            assert nobs == G * 16
            want = snapkv_max_score([list(st.rq) for st in u.heads],
                                    bf16_to_f64(np.stack(u.K)), u.pos, 1e6, d)
            assert np.allclose(got, want, rtol=1e-12, atol=0)
        u.evict(t - 1)


def snapkv_mean_score(heads_recent, K_vals, k_pos, theta, d):
    """Recent-window mean score (eq. 6 of the notes) averaged over the query
    heads of the group as well, written as explicit loops: every observation
    row contributes its softmax weight (0 for keys it cannot access)."""
    L = len(K_vals)
    total = [0.0] * L
    rows = 0
    for recent in heads_recent:
        for q, tau in recent:
            rows += 1
            qr = rope(bf16_to_f64(q), tau, theta)
            acc = [j for j in range(L) if k_pos[j] <= tau]
            logit = {j: float(qr @ K_vals[j]) / math.sqrt(d) for j in acc}
            mx = max(logit.values())
            z = math.fsum(math.exp(v - mx) for v in logit.values())
            for j in acc:
                total[j] += math.exp(logit[j] - mx) / z
    return np.array(total) / rows


def test_mean_pool_zero_beacons_is_the_recent_window_mean_formula():
    G, d = 2, 128
    u = UnitOracle(group=G, d=d, theta=1e6, budget=40, prefix=4, recent=8, fps_cap=16,
                   fps_keep=0, pool="mean")
    g = torch.Generator().manual_seed(12)
    t = 0
    for rnd in range(2):
        while len(u.K) < 56:
            u.append_kv(to_bits(torch.randn(d, generator=g).to(torch.bfloat16)),
                        to_bits(torch.randn(d, generator=g).to(torch.bfloat16)), t)
            u.append_queries(to_bits(torch.randn(G, d, generator=g).to(torch.bfloat16)), t)
            t += 1
        if rnd == 1:
            got, nobs = u.scores(t - 1)
            want = snapkv_mean_score([list(st.rq) for st in u.heads],
                                     bf16_to_f64(np.stack(u.K)), u.pos, 1e6, d)
            assert nobs == G * 16
            assert np.allclose(got, want, rtol=1e-12, atol=0)
        u.evict(t - 1)


@pytest.mark.parametrize("seed", range(5))
def test_mean_pool_scores_sum_to_one_and_bound_the_max(seed):
    """Each softmax row sums to 1 over its accessible keys, so the mean over
    rows sums to 1 over the cache; the mean never exceeds the max, and with
    one row the two poolings coincide."""
    g = np.random.default_rng(seed)
    R, L, d = int(g.integers(1, 12)), int(g.integers(5, 60)), 16
    Q, K = g.standard_normal((R, d)), g.standard_normal((L, d))
    qpos = g.integers(L // 2, L, size=R)
    W = attention_weights(Q, qpos, K, np.arange(L))
    mp = mean_pool(W)
    assert math.isclose(float(mp.sum()), 1.0, rel_tol=1e-12)
    assert np.all(mp <= max_pool(W) + 1e-15)
    assert np.allclose(mean_pool(W[:1]), max_pool(W[:1]), rtol=0, atol=0)


def test_coverage_closed_forms():
    """A member of the set covers itself (cosine 1 up to the float64 square
    root), its negation scores -1, an orthogonal query 0, a zero query 0, a
    scaled copy 1; the max is over the whole set; an empty set gives -inf."""
    e = np.eye(128)[:3]
    obs = [bf16_bits(e[0]), bf16_bits(e[1] * 2.0)]
    fut = [bf16_bits(e[0]), bf16_bits(-e[0]), bf16_bits(e[2]), bf16_bits(np.zeros(128)),
           bf16_bits(e[1] * 0.5), bf16_bits(e[0] + e[1])]
    got = coverage(obs, fut)
    assert got[0] == 1.0 and got[1] == 0.0 and got[2] == 0.0 and got[3] == 0.0
    assert got[4] == 1.0
    assert math.isclose(got[5], 1 / math.sqrt(2), rel_tol=1e-15)
    assert coverage([bf16_bits(-e[0])], [bf16_bits(e[0])]) == [-1.0]
    assert coverage([], [bf16_bits(e[0])]) == [-math.inf]


@pytest.mark.parametrize("seed", range(5))
def test_coverage_matches_rational_brute_force(seed):
    """Against exact rational arithmetic: the max cosine is attained by the
    row with the largest G_qo / sqrt(G_oo), and its float64 value is the
    correctly rounded quotient of the exact dot products."""
    obs = rand_bits((7, 128), seed=200 + seed)
    fut = rand_bits((5, 128), seed=300 + seed)
    got = coverage(obs, fut)
    for f, c in zip(fut, got):
        fq = [Fraction(float(v)) for v in bf16_to_f64(f)]
        gqq = sum(x * x for x in fq)
        best = None
        for o in obs:
            ov = [Fraction(float(v)) for v in bf16_to_f64(o)]
            goo = sum(x * x for x in ov)
            gqo = sum(x * y for x, y in zip(fq, ov))
            val = float(gqo) / math.sqrt(float(gqq) * float(goo))
            best = val if best is None else max(best, val)
        assert c == best


@pytest.mark.parametrize("P", [1, 3, 4, 6, 8])
def test_prefill_of_a_short_prompt_equals_streaming_appends(P):
    """While the earlier prompt queries fit in fps_keep no FPS runs either
    way, so prefill must leave exactly the state of P single-step appends
    (beacons = the spilled queries in order, recents = the last n_rq)."""
    mk = lambda: UnitOracle(group=3, d=128, theta=1e6, budget=20, prefix=2, recent=4,
                            fps_cap=8, fps_keep=4)
    a, b = mk(), mk()
    q = rand_bits((P, 3, 128), seed=400 + P)   # n_rq = 4, so at most fps_keep = 4 older queries
    for t in range(P):
        a.append_queries(q[t], 100 + t)
    b.prefill([q[:, h] for h in range(3)], 100)
    for sa, sb in zip(a.heads, b.heads):
        assert [r.tobytes() for r in sa.bq] == [r.tobytes() for r in sb.bq]
        assert [(r.tobytes(), p) for r, p in sa.rq] == [(r.tobytes(), p) for r, p in sb.rq]


@pytest.mark.parametrize("seed", range(6))
def test_prefill_beacons_are_brute_force_fps_of_the_older_queries(seed):
    """The beacons and trace are the greedy rule re-derived by brute force
    (max-cosine-to-set recomputed from rational Gram entries) over the
    prompt's queries older than the recent window."""
    g = np.random.default_rng(seed)
    P, n_rq, keep = int(g.integers(20, 36)), 5, 6
    u = UnitOracle(group=1, d=128, theta=1e6, budget=20, prefix=2, recent=4, fps_cap=keep + n_rq,
                   fps_keep=keep)
    q = rand_bits((P, 128), seed=500 + seed)
    u.prefill([q], 7)
    want = fps_brute(q[:P - n_rq], keep)
    assert u.heads[0].trace == want
    assert [r.tobytes() for r in u.heads[0].bq] == [q[i].tobytes() for i in sorted(want)]
    assert [p for _, p in u.heads[0].rq] == list(range(7 + P - n_rq, 7 + P))


# ---------------------------------------------------------------------------- keep set

@pytest.mark.parametrize("seed", range(20))
def test_select_keep_matches_full_sort(seed):
    g = np.random.default_rng(seed)
    L = int(g.integers(30, 300))
    prefix, recent = int(g.integers(0, 6)), int(g.integers(0, 20))
    budget = int(g.integers(prefix + recent, L))
    score = g.random(L).round(2)                  # plenty of exact ties
    kept = select_keep(score, L, prefix, recent, budget)
    assert len(kept) == budget and kept == sorted(set(kept))
    assert set(range(prefix)) <= set(kept) and set(range(L - recent, L)) <= set(kept)
    cands = np.array([j for j in range(prefix, L - recent)])
    order = cands[np.lexsort((cands, -score[cands]))]
    want = sorted(set(range(prefix)) | set(range(L - recent, L))
                  | set(order[:budget - prefix - recent].tolist()))
    assert kept == want


def test_compaction_is_a_bytewise_gather():
    u = UnitOracle(group=1, d=128, theta=1e6, budget=20, prefix=2, recent=4, fps_cap=4,
                   fps_keep=2)
    rows = rand_bits((28, 128), seed=9)
    vals = rand_bits((28, 128), seed=10)
    for t in range(28):
        u.append_kv(rows[t], vals[t], t)
        u.append_queries(rand_bits((1, 128), seed=100 + t), t)
    res = u.evict(27)
    assert np.array_equal(np.stack(u.K), rows[res.kept])
    assert np.array_equal(np.stack(u.V), vals[res.kept])
    assert u.pos == res.kept


def test_order_free_layout_golden():
    gd = read_golden("order_free_layout.txt")
    score = np.array([float(x) for x in gd["scores"].split(",")])
    L, budget, prefix, recent = (int(gd[k]) for k in ("L", "budget", "prefix", "recent"))
    kept = select_keep(score, L, prefix, recent, budget)
    assert kept == [int(x) for x in gd["kept"].split(",")]
    layout = order_free_layout(kept, budget)
    assert layout == [int(x) for x in gd["layout"].split(",")]
    assert sum(1 for i, j in enumerate(layout) if i != j) == int(gd["moved"])


@pytest.mark.parametrize("seed", range(20))
def test_order_free_layout_properties(seed):
    """Against the definition restated slot by slot: kept slots below the budget
    stay, holes take the tail in order, and the layout is the keep set."""
    g = np.random.default_rng(seed)
    L = int(g.integers(20, 400))
    budget = int(g.integers(1, L))
    kept = sorted(g.choice(L, size=budget, replace=False).tolist())
    layout = order_free_layout(kept, budget)
    assert sorted(layout) == kept
    tail = iter(j for j in kept if j >= budget)
    moved = 0
    for i in range(budget):
        if i in kept:
            assert layout[i] == i
        else:
            assert layout[i] == next(tail)
            moved += 1
    assert moved == sum(1 for j in kept if j >= budget) <= L - budget


@pytest.mark.parametrize("recent,period", [(4, 6), (6, 6), (0, 5)])
def test_order_free_stream_keeps_the_same_tokens(recent, period):
    """With the recent window inside the appended tail (recent <= period), an
    order-free stream keeps exactly the tokens (by position), the K/V rows and
    the FPS picks of the sorted stream at every eviction; only the slot layout
    differs. Slot-based prefix/recent protection and masking therefore keep
    their positional meaning after holes are filled from the tail."""
    budget, prefix = 24, 2
    mk = lambda of: UnitOracle(group=2, d=128, theta=1e6, budget=budget, prefix=prefix,
                               recent=recent, fps_cap=6, fps_keep=3, order_free=of)
    a, b = mk(False), mk(True)
    keys, vals = rand_bits((200, 128), seed=31), rand_bits((200, 128), seed=32)
    qs = rand_bits((200, 2, 128), seed=33)
    evictions = 0
    for t in range(200):
        for u in (a, b):
            u.append_kv(keys[t], vals[t], t)
            u.append_queries(qs[t], t)
        if len(a.K) == budget + period:
            ra, rb = a.evict(t), b.evict(t)
            evictions += 1
            assert ra.traces == rb.traces
            assert sorted(a.pos) == sorted(b.pos)
            by_pos = {p: (k.tobytes(), v.tobytes()) for p, k, v in zip(b.pos, b.K, b.V)}
            assert all(by_pos[p] == (k.tobytes(), v.tobytes()) for p, k, v in zip(a.pos, a.K, a.V))
            assert a.pos == sorted(a.pos)
            assert sum(1 for i, j in enumerate(rb.layout) if i != j) <= period
    assert evictions >= 10


# ---------------------------------------------------------------------------- state machine

class Alg2Head:
    """Algorithm 2 of the notes, in its own single-buffer form: the buffer
    collects queries (FPS when it reaches the cap) until the cache reaches
    B_max - n_recent; then it is frozen as the beacons and the next n_recent
    queries are collected with their positions; after the eviction
    FPS(beacons + recents) is the new buffer, frozen again at once."""

    def __init__(self, cap, keep):
        self.cap, self.keep = cap, keep
        self.buf, self.beacons, self.recents = [], None, []

    def push(self, q, tau):
        if self.beacons is None:
            self.buf.append(q)
            if len(self.buf) >= self.cap:
                _, k = fps(bf16_to_f64(np.stack(self.buf)), self.keep)
                self.buf = [self.buf[i] for i in k]
        else:
            self.recents.append((q, tau))

    def freeze(self):
        self.beacons, self.recents = list(self.buf), []

    def after_evict(self):
        X = self.beacons + [q for q, _ in self.recents]
        if len(X) > self.keep:
            _, k = fps(bf16_to_f64(np.stack(X)), self.keep)
            X = [X[i] for i in k]
        self.buf, self.beacons, self.recents = X, None, []


def test_ring_state_machine_equals_algorithm_2():
    G, d, budget, period, cap, keep = 2, 16, 48, 16, 32, 16
    u = UnitOracle(group=G, d=d, theta=1e4, budget=budget, prefix=4, recent=16,
                   fps_cap=cap, fps_keep=keep)
    alg = [Alg2Head(cap, keep) for _ in range(G)]
    g = torch.Generator().manual_seed(5)
    L, evictions = 0, 0
    for t in range(260):
        q = to_bits(torch.randn(G, d, generator=g).to(torch.bfloat16))
        u.append_kv(np.zeros(d, np.uint16), np.zeros(d, np.uint16), t)
        u.append_queries(q, t)
        L += 1
        for h in range(G):
            alg[h].push(q[h], t)
        if L == budget + period - (cap - keep):
            for a in alg:
                if a.beacons is None:
                    a.freeze()
        if L == budget + period:
            for h in range(G):
                st = u.heads[h]
                assert len(st.bq) == len(alg[h].beacons)
                assert all(np.array_equal(x, y) for x, y in zip(st.bq, alg[h].beacons))
                assert [p for _, p in st.rq] == [p for _, p in alg[h].recents] \
                    == list(range(t - 15, t + 1))
                assert all(np.array_equal(x, y) for (x, _), (y, _) in zip(st.rq, alg[h].recents))
            u.evict(t)
            for a in alg:
                a.after_evict()
                a.freeze()
            L = budget
            evictions += 1
    assert evictions >= 10


# ---------------------------------------------------------------------------- byte model

def test_kv_byte_model_matches_pages_motivating_example():
    gd = read_golden("kv_bytes_qwen3_4b.txt")
    per_tok = kv_bytes_per_token(int(gd["layers"]), int(gd["kv_heads"]), int(gd["d"]))
    assert per_tok == int(gd["bytes_per_token"])
    total = per_tok * int(gd["tokens"]) * int(gd["batch"])
    assert total == int(gd["total_bytes"]) and total > int(gd["lower_bound_gb"]) * 1e9


def test_observation_rows_rotate_beacons_to_t_and_recents_to_tau():
    """Q_obs of the notes' §2.3: beacons at the eviction step t, recents at their
    own positions. With d = 2, RoPE at position p is the plane rotation by p."""
    u = UnitOracle(group=1, d=2, theta=1e4, budget=4, prefix=0, recent=0, fps_cap=4, fps_keep=2)
    g = np.random.default_rng(4)
    for tau in range(7):
        u.append_queries(bf16_bits(g.standard_normal((1, 2))), tau)
    st = u.heads[0]
    assert len(st.bq) == 3 and [p for _, p in st.rq] == [5, 6]
    t = 9
    rows, pos = u.observation(t)

    def rot(x, a):
        return [x[0] * math.cos(a) - x[1] * math.sin(a), x[1] * math.cos(a) + x[0] * math.sin(a)]

    want = [rot(bf16_to_f64(q), t) for q in st.bq] + [rot(bf16_to_f64(q), p) for q, p in st.rq]
    assert np.allclose(rows, want, rtol=0, atol=1e-14)
    assert list(pos) == [t, t, t, 5, 6]
