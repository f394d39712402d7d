"""The float32 error bound behind the FPS kernel's decisions, checked on the CPU.

The eviction-time FPS kernel forms each head's Gram on the tensor cores: the
128 products of two bf16 rows are exact, but the order of the 127 additions
and their roundings are the hardware's. Its filters therefore assume only
float32 precision at every addition, in any rounding direction, with products
or partial sums below 2^-126 possibly flushed to zero. From that, the cosine
c = (G_ij r_i) r_j, with r = rsqrt(G_ii) to 2 ulp, lies within 3.2e-5 of the
float64 cosine (BeaconKV reading notes §2.2, Algorithm 1: cosine similarity of
pre-RoPE queries), and the filters allow 4e-5. Rows enter that Gram as loaded
when every 8-element piece is zero or has its largest magnitude in
[2^-40, 2^21).

These tests build such rows at both ends of that range. Each pair's products
are summed in a random order or by decreasing or increasing magnitude. Every
addition is rounded in a random direction, always up or always down, and
results below 2^-126 are flushed at random. Each Gram entry is checked
against its own bound. The cosine uses an rsqrt perturbed by up to 2 ulp and
is compared with the oracle's float64 cosine (exact Gram, IEEE float64 divide
and square root). A control shows the test can fail: rows below the range
lose their Gram to flushing.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import cosine_matrix, gram_exact

COS_BOUND = 3.2e-5      # the bound the kernel derives; its filters use 4e-5
TINY = 2.0 ** -126      # smallest normal float32


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Rounds to bf16 (nearest even) and returns the exact values as float64."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def pieces_in_range(row: np.ndarray) -> bool:
    """Every 8-element piece is zero or has its largest magnitude in [2^-40, 2^21)."""
    m = np.abs(row).reshape(-1, 8).max(axis=1)
    return bool(np.all((m == 0) | ((m >= 2.0 ** -40) & (m < 2.0 ** 21))))


def round_f32(s: np.ndarray, up: np.ndarray) -> np.ndarray:
    """s (float64) rounded to float32 downwards where ~up, upwards where up."""
    f = s.astype(np.float32)
    fd = f.astype(np.float64)
    lower = np.where(fd > s, np.nextafter(f, np.float32(-np.inf)), f)
    upper = np.where(fd < s, np.nextafter(f, np.float32(np.inf)), f)
    return np.where(up, upper, lower).astype(np.float64)


def flush(x: np.ndarray, on: np.ndarray) -> np.ndarray:
    return np.where(on & (np.abs(x) < TINY), 0.0, x)


def gram_f32_any_order(X: np.ndarray, rng: np.random.Generator, flush_p: float = 0.5,
                       order: str = "random", direction: str = "random") -> np.ndarray:
    """Every entry of X X^T as a float32 sum of its exact products: in a random
    order, or by decreasing or increasing magnitude; each addition rounded in
    a random direction, or always up, or always down; products and partial
    sums below 2^-126 flushed with probability flush_p per entry."""
    n, d = X.shape
    ii, jj = np.triu_indices(n)
    prods = X[ii] * X[jj]                                    # exact in float64
    key = {"random": rng.random(prods.shape), "desc": -np.abs(prods), "asc": np.abs(prods)}[order]
    prods = np.take_along_axis(prods, np.argsort(key, axis=1, kind="stable"), axis=1)
    fl = rng.random(len(ii)) < flush_p
    prods = flush(prods, fl[:, None])
    acc = np.zeros(len(ii))
    for k in range(d):
        up = {"random": rng.random(len(ii)) < 0.5, "up": np.ones(len(ii), bool),
              "down": np.zeros(len(ii), bool)}[direction]
        acc = flush(round_f32(acc + prods[:, k], up), fl)
    G = np.zeros((n, n))
    G[ii, jj] = acc
    G[jj, ii] = acc
    return G


def cos_f32(G32: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """c_ij = (G_ij * r_i) * r_j in float32, r_i = rsqrt(G_ii) off by up to 2 ulp."""
    diag = np.diag(G32).astype(np.float32)
    d64 = diag.astype(np.float64)
    r = np.divide(1.0, np.sqrt(d64), out=np.zeros_like(d64), where=d64 > 0).astype(np.float32)
    for _ in range(2):
        step = rng.integers(-1, 2, size=r.shape)
        r = np.where(step > 0, np.nextafter(r, np.float32(np.inf)),
                     np.where(step < 0, np.nextafter(r, np.float32(0)), r))
    r = np.where(diag > 0, r, np.float32(0))
    g = G32.astype(np.float32)
    return ((g * r[:, None]).astype(np.float32) * r[None, :]).astype(np.float64)


def edge_rows(rng: np.random.Generator, n: int) -> np.ndarray:
    """bf16 rows at the ends of the as-loaded range: whole rows near 2^21 and
    near 2^-40, rows mixing pieces at both ends, near-duplicates, negated
    copies, zero pieces and a zero row, all satisfying the range test."""
    rows = []
    while len(rows) < n:
        kind = len(rows) % 6
        base = rng.standard_normal(128)
        if kind == 0:      # largest component just below 2^21
            x = base / np.abs(base).max() * (2.0 ** 21) * (1 - 2.0 ** -8)
        elif kind == 1:    # every piece's largest component just above 2^-40
            p = base.reshape(-1, 8)
            x = (p / np.abs(p).max(axis=1, keepdims=True) * 2.0 ** -40 * (1 + rng.random((16, 1)))).ravel()
        elif kind == 2:    # pieces alternating between the two ends
            p = base.reshape(-1, 8)
            s = np.where(np.arange(16)[:, None] % 2 == 0, 2.0 ** 20, 2.0 ** -39)
            x = (p / np.abs(p).max(axis=1, keepdims=True) * s).ravel()
        elif kind == 3 and rows:    # near-duplicate of an earlier row
            x = rows[rng.integers(len(rows))] * (1 + 2.0 ** -7 * rng.standard_normal(128))
        elif kind == 4 and rows:    # negated earlier row with zeroed pieces
            x = -rows[rng.integers(len(rows))].copy()
            x.reshape(-1, 8)[rng.random(16) < 0.25] = 0.0
        else:
            x = base * 2.0 ** rng.integers(-38, 19)
        x = to_bf16(x)
        if pieces_in_range(x):
            rows.append(x)
    rows[-1] = np.zeros(128)
    return np.stack(rows)


def max_cos_error(X: np.ndarray, rng: np.random.Generator, flush_p: float = 0.5, **mode) -> float:
    C64 = np.array(cosine_matrix(gram_exact(X)))
    C32 = cos_f32(gram_f32_any_order(X, rng, flush_p, **mode), rng)
    return float(np.max(np.abs(C32 - C64)))


MODES = [dict(order=o, direction=d) for o in ("random", "desc", "asc") for d in ("random", "up", "down")]


def test_gram_entries_stay_within_their_bound():
    """|G32 - G| <= 127 * 2^-23 * sum_k |x_ik x_jk| + 255 * 2^-126 for every
    entry, whatever the order and the rounding directions."""
    rng = np.random.default_rng(5)
    worst = 0.0
    for mode in MODES:
        X = edge_rows(rng, 30)
        G = np.array(gram_exact(X))
        bound = 127 * 2.0 ** -23 * (np.abs(X) @ np.abs(X).T) + 255 * TINY
        err = np.abs(gram_f32_any_order(X, rng, 0.5, **mode) - G)
        assert np.all(err <= bound), mode
        worst = max(worst, float(np.max(err / bound)))
    assert worst > 1e-3  # the one-direction sums do move the Gram


def test_rows_used_as_loaded_stay_within_the_cosine_bound():
    rng = np.random.default_rng(20261202)
    worst = {}
    for mode in MODES:
        for _ in range(2):
            X = edge_rows(rng, 36)
            key = (mode["order"], mode["direction"])
            worst[key] = max(worst.get(key, 0.0), max_cos_error(X, rng, **mode))
    assert max(worst.values()) <= COS_BOUND, worst
    assert worst[("desc", "up")] > worst[("random", "random")]


def test_round_f32_takes_the_requested_direction():
    s = np.array([1.0 + 2.0 ** -30, -(1.0 + 2.0 ** -30), 3.0])
    down = round_f32(s, np.array([False, False, False]))
    up = round_f32(s, np.array([True, True, True]))
    assert down[0] == 1.0 and up[0] == 1.0 + 2.0 ** -23
    assert down[1] == -(1.0 + 2.0 ** -23) and up[1] == -1.0
    assert down[2] == up[2] == 3.0


def test_rows_below_the_range_can_lose_their_gram_to_flushing():
    """Control: rows whose components all lie near 2^-64 have products near
    2^-128; flushed, the float32 Gram loses them and the cosine is far off, so
    the range test is what keeps the bound."""
    rng = np.random.default_rng(7)
    base = rng.standard_normal((4, 128))
    X = to_bf16(np.concatenate([base, base + 0.01 * rng.standard_normal((4, 128))]) * 2.0 ** -64)
    assert not any(pieces_in_range(x) for x in X)
    assert max_cos_error(X, rng, flush_p=1.0) > 1e-3
