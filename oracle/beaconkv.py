"""fp64 CPU oracle of BeaconKV's periodic KV-cache eviction step.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
bench.py's CPU-baseline legs, never by the product path.

Source. The method is stated on the page "BeaconKV：用历史查询代表保护长推理的远程回看"
(reading notes on the BeaconKV paper, liuzhao09.github.io), cited below as
"BeaconKV reading notes" with its section and equation; the rcap.io summary
"BeaconKV: Key-Value Cache Compression Guided by Beacon Queries" gives the
32 -> 16 buffer sizes.

Everything is plain loops or single library primitives (a numpy matmul, an
exp, a sort, math.fsum) in float64 on the exact values of the bf16 inputs.
Inputs arrive as numpy uint16 arrays holding bf16 bit patterns.

Readings taken where the pages are silent (each one is listed in the design
notes with its reason):
  * one query buffer per query head; a unit is one (sequence, layer, KV head)
    and owns its G query heads' buffers;
  * RoPE is rotate-half on pairs (i, i + d/2) with inv_freq_i = theta^(-2i/d);
  * the exact Gram entry is the exactly rounded sum of exact products;
  * the mean cosine includes j = i and is summed left to right in fp64;
  * every argmin / top-k tie goes to the lowest index / lowest slot;
  * a zero vector has cosine 0 with everything;
  * a recent observation row at position tau sees only keys at positions
    <= tau (accessible keys, eq. 4); beacons, rotated to t, see every key.
"""

from __future__ import annotations

import math
from collections import deque
from dataclasses import dataclass, field

import numpy as np


# ----------------------------------------------------------------------------
# values


def bf16_to_f64(bits) -> np.ndarray:
    """Exact float64 values of bf16 bit patterns (bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# RoPE re-alignment (BeaconKV reading notes, §2.3, the Q_obs equation)


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotary position encoding of vector(s) x at absolute position(s) pos.

    Rotate-half convention: for i < d/2 the pair (x_i, x_{i+d/2}) is rotated
    by the angle pos * theta^(-2i/d):
        out_i       = x_i * cos - x_{i+d/2} * sin
        out_{i+d/2} = x_{i+d/2} * cos + x_i * sin
    `pos` broadcasts against the leading axes of x.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    inv_freq = theta ** (-2.0 * np.arange(h, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty(np.broadcast_shapes(x.shape, c.shape[:-1] + (d,)), dtype=np.float64)
    out[..., :h] = x[..., :h] * c - x[..., h:] * s
    out[..., h:] = x[..., h:] * c + x[..., :h] * s
    return out


# ----------------------------------------------------------------------------
# farthest-point sampling (BeaconKV reading notes, §2.2, Algorithm 1)


def exact_dot(a, b) -> float:
    """sum_k a_k b_k of bf16-valued vectors, rounded once to float64.

    Each product of two bf16 values has at most 16 significant bits and an
    exponent far inside float64's range, so it is exact in float64; math.fsum
    then returns the correctly rounded value of their exact sum.
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return math.fsum((a * b).tolist())


def gram_exact(X) -> list[list[float]]:
    """G[i][j] = exact_dot(X[i], X[j]) for the rows of X."""
    X = np.asarray(X, dtype=np.float64)
    n = X.shape[0]
    G = [[0.0] * n for _ in range(n)]
    for i in range(n):
        for j in range(i, n):
            G[i][j] = G[j][i] = exact_dot(X[i], X[j])
    return G


def cosine_matrix(G) -> list[list[float]]:
    """cos(q_i, q_j) = G_ij / sqrt(G_ii * G_jj) in IEEE float64; 0 if either norm is 0."""
    n = len(G)
    C = [[0.0] * n for _ in range(n)]
    for i in range(n):
        for j in range(n):
            if G[i][i] == 0.0 or G[j][j] == 0.0:
                C[i][j] = 0.0
            else:
                C[i][j] = G[i][j] / math.sqrt(G[i][i] * G[j][j])
    return C


def _argmin_lowest(values, allowed) -> int:
    best = -1
    for j in allowed:
        if best < 0 or values[j] < values[best]:
            best = j
    return best


def fps(X, m: int) -> tuple[list[int], list[int]]:
    """Farthest-point sampling of m rows of X by cosine similarity.

    Algorithm 1 of the BeaconKV reading notes (§2.2):
      a_i = (1/N) sum_{j=1..N} cos(q_i, q_j),  p = argmin_i a_i,  I = {p},
      S_j = cos(q_j, q_p);
      repeat: r = argmin_{j not in I} S_j,  I <- I + {r},
              S_j <- max(S_j, cos(q_j, q_r))      until |I| = m.
    Returns (trace, kept): the picks in pick order and the same indices
    sorted ascending. With N <= m every row is kept and the trace is 0..N-1.
    """
    X = np.asarray(X, dtype=np.float64)
    n = X.shape[0]
    if n <= m:
        return list(range(n)), list(range(n))
    if m == 0:
        return [], []
    C = cosine_matrix(gram_exact(X))
    a = []
    for i in range(n):
        acc = 0.0
        for j in range(n):
            acc = acc + C[i][j]
        a.append(acc / n)
    p = _argmin_lowest(a, range(n))
    picked = [p]
    chosen = [False] * n
    chosen[p] = True
    S = [C[j][p] for j in range(n)]
    while len(picked) < m:
        r = _argmin_lowest(S, [j for j in range(n) if not chosen[j]])
        picked.append(r)
        chosen[r] = True
        S = [max(S[j], C[j][r]) for j in range(n)]
    return picked, sorted(picked)


# ----------------------------------------------------------------------------
# scoring (BeaconKV reading notes, §2.1 eqs. 4-5 and §2.3 eq. 7)


def attention_weights(Q, q_pos, K, k_pos) -> np.ndarray:
    """W[r, j] = exp(q_r.k_j/sqrt d) / sum_{l accessible} exp(q_r.k_l/sqrt d).

    Key j is accessible from row r when its position k_pos[j] <= q_pos[r];
    inaccessible entries are 0. Q are the already-rotated observation rows.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = Q.shape[1]
    logits = (Q @ K.T) / math.sqrt(d)
    access = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    logits = np.where(access, logits, -np.inf)
    shift = logits.max(axis=1, keepdims=True)
    e = np.where(access, np.exp(logits - shift), 0.0)
    return e / e.sum(axis=1, keepdims=True)


def max_pool(W) -> np.ndarray:
    """Score[j] = max over every observation row (all query heads of the group) of W[., j]."""
    return np.asarray(W).max(axis=0)


def mean_pool(W) -> np.ndarray:
    """Score[j] = the mean of W[., j] over every observation row, the mean
    aggregation of BeaconKV reading notes §2.1 eq. 6 applied over queries and
    heads together (Table 2 compares the two aggregations over both at once).
    Inaccessible entries are 0 and count in the denominator."""
    W = np.asarray(W, dtype=np.float64)
    return W.sum(axis=0) / W.shape[0]


def coverage(obs, future) -> list[float]:
    """Future-query coverage (BeaconKV reading notes §3.2, Figure 6): for each
    future query, the largest cosine between it and any row of the observation
    set, with the cosine of cosine_matrix (exact dot products, IEEE float64).
    -inf for an empty observation set."""
    obs = [bf16_to_f64(o) for o in obs]
    out = []
    for q in future:
        qv = bf16_to_f64(q)
        gqq = exact_dot(qv, qv)
        best = -math.inf
        for o in obs:
            goo = exact_dot(o, o)
            c = 0.0 if gqq == 0.0 or goo == 0.0 else exact_dot(qv, o) / math.sqrt(gqq * goo)
            best = max(best, c)
        out.append(best)
    return out


# ----------------------------------------------------------------------------
# keep set and compaction (BeaconKV reading notes, §2.3 eq. 8)


def select_keep(score, L: int, prefix: int, recent: int, budget: int) -> list[int]:
    """I_final = Sort(I_keep + TopK(Score, k_sel, exclude=I_keep)) as 0-based slots.

    I_keep = prefix slots [0, prefix) and the recent window [L-recent, L);
    k_sel = budget - |I_keep|; the top-k orders by score descending and then
    by slot ascending (lowest slot wins a tie).
    """
    keep = set(range(min(prefix, L))) | set(range(max(L - recent, 0), L))
    cands = [j for j in range(L) if j not in keep]
    k_sel = budget - len(keep)
    order = sorted(cands, key=lambda j: (-float(score[j]), j))
    return sorted(keep | set(order[:k_sel]))


def order_free_layout(kept, budget: int) -> list[int]:
    """Slot layout of an order-free compaction, a relaxation of eq. 8's Sort.

    The kept set is the one eq. 8 selects (`kept`, any order). Instead of
    gathering it in slot order, every kept slot below `budget` stays where it
    is and the dropped slots below `budget` (the holes, ascending) receive the
    kept slots at or above `budget` (ascending). Returns `layout`: after the
    compaction slot i holds the row that was in slot layout[i]. Exactly as many
    rows move as there are holes.
    """
    ks = sorted(int(j) for j in kept)
    inside = set(j for j in ks if j < budget)
    holes = [i for i in range(budget) if i not in inside]
    tail = [j for j in ks if j >= budget]
    assert len(holes) == len(tail), "a keep set of `budget` slots has one tail slot per hole"
    layout = list(range(budget))
    for i, j in zip(holes, tail):
        layout[i] = j
    return layout


# ----------------------------------------------------------------------------
# the per-unit state machine (BeaconKV reading notes, §2.2 eq. 9 and Algorithm 2)


@dataclass
class HeadState:
    """One query head's pre-RoPE observation state: beacons Bq and recents R."""
    bq: list = field(default_factory=list)              # uint16 rows, oldest first
    rq: deque = field(default_factory=deque)            # (uint16 row, position), oldest first
    trace: list = field(default_factory=list)           # picks of the last FPS call


@dataclass
class EvictResult:
    kept: list          # the keep set this oracle selected, ascending
    score: np.ndarray
    obs_rows: int
    traces: list
    layout: list = field(default_factory=list)   # source slot of each slot after compaction


class UnitOracle:
    """One eviction unit: a (sequence, layer, KV head) cache slice and the G
    query heads that share it.

    append_kv / append_queries follow one decode step; evict runs the step at
    time t. Buffers: B_Q^min = fps_keep beacons, B_Q^max = fps_cap, so the
    recent-query ring holds n_rq = fps_cap - fps_keep entries (eq. 9).
      push(q, tau): R <- R + <q, tau>; if |R| > n_rq the oldest query moves to
                    the end of Bq; if |Bq| >= fps_cap then Bq <- FPS(Bq, fps_keep).
      evict(t):     observation rows RoPE(Bq, t) and RoPE(q, tau) for <q, tau>
                    in R, per head; score, keep, compact; then per head
                    Bq <- FPS(Bq + R, fps_keep) and R <- empty (Algorithm 2).
    With order_free, the compaction keeps the same set but in the layout of
    order_free_layout (holes below the budget filled from the tail); keys
    carry their positions, so later masking is unchanged. pool = "mean"
    scores with mean_pool instead of max_pool (Table 2's ablation).
    """

    def __init__(self, group: int, d: int, theta: float, budget: int, prefix: int,
                 recent: int, fps_cap: int, fps_keep: int, order_free: bool = False,
                 pool: str = "max"):
        assert pool in ("max", "mean")
        self.order_free = order_free
        self.pool = pool
        self.group, self.d, self.theta = group, d, theta
        self.budget, self.prefix, self.recent = budget, prefix, recent
        self.fps_cap, self.fps_keep = fps_cap, fps_keep
        self.n_rq = fps_cap - fps_keep
        self.heads = [HeadState() for _ in range(group)]
        self.K: list[np.ndarray] = []
        self.V: list[np.ndarray] = []
        self.pos: list[int] = []

    # -- decode-side updates ------------------------------------------------
    def append_kv(self, k_row, v_row, pos: int) -> None:
        self.K.append(np.asarray(k_row, dtype=np.uint16).copy())
        self.V.append(np.asarray(v_row, dtype=np.uint16).copy())
        self.pos.append(int(pos))

    def append_queries(self, q_rows, tau: int) -> None:
        for h, st in enumerate(self.heads):
            st.rq.append((np.asarray(q_rows[h], dtype=np.uint16).copy(), int(tau)))
            if len(st.rq) > self.n_rq:
                st.bq.append(st.rq.popleft()[0])
            if len(st.bq) >= self.fps_cap:
                st.trace, keep = fps(bf16_to_f64(np.stack(st.bq)), self.fps_keep)
                st.bq = [st.bq[i] for i in keep]

    # -- eviction -------------------------------------------------------------
    def observation(self, t: int) -> tuple[np.ndarray, np.ndarray]:
        """Rotated observation rows (fp64) and their positions, head by head."""
        rows, poss = [], []
        for st in self.heads:
            for q in st.bq:
                rows.append(rope(bf16_to_f64(q), t, self.theta))
                poss.append(t)
            for q, tau in st.rq:
                rows.append(rope(bf16_to_f64(q), tau, self.theta))
                poss.append(tau)
        if not rows:
            return np.zeros((0, self.d)), np.zeros((0,), dtype=np.int64)
        return np.stack(rows), np.asarray(poss, dtype=np.int64)

    def scores(self, t: int) -> tuple[np.ndarray, int]:
        Q, qpos = self.observation(t)
        L = len(self.K)
        if Q.shape[0] == 0:
            return np.zeros(L), 0
        W = attention_weights(Q, qpos, bf16_to_f64(np.stack(self.K)), np.asarray(self.pos))
        return (mean_pool(W) if self.pool == "mean" else max_pool(W)), Q.shape[0]

    def evict(self, t: int, kept_override=None, score=None) -> EvictResult:
        """One eviction at time t. `kept_override`, when given, is a keep set the
        caller has already checked against this oracle's own one (a different
        but equally valid choice inside the score tie band); compaction and the
        following state then use it. `score`, when given, is this unit's
        scores(t) computed just before (saves recomputing it)."""
        L = len(self.K)
        if score is None:
            score, nobs = self.scores(t)
        else:
            nobs = self.observation(t)[0].shape[0]
        kept = select_keep(score, L, self.prefix, self.recent, self.budget)
        use = sorted(kept_override) if kept_override is not None else kept
        layout = order_free_layout(use, self.budget) if self.order_free else use
        self.K = [self.K[i] for i in layout]
        self.V = [self.V[i] for i in layout]
        self.pos = [self.pos[i] for i in layout]
        traces = []
        for st in self.heads:
            X = st.bq + [q for q, _ in st.rq]
            if len(X) > self.fps_keep:
                st.trace, keep = fps(bf16_to_f64(np.stack(X)), self.fps_keep)
                st.bq = [X[i] for i in keep]
            else:
                st.trace = list(range(len(X)))
                st.bq = X
            st.rq.clear()
            traces.append(list(st.trace))
        return EvictResult(kept=kept, score=score, obs_rows=nobs, traces=traces, layout=layout)

    def prefill(self, q_prompt, first_step: int) -> None:
        """Initial observation state from a prompt (BeaconKV reading notes §2.2:
        at prefill the first representatives are sampled from the input
        queries). Per head, of the P prompt queries (positions first_step ...
        first_step + P - 1), the last min(n_rq, P) become the recent queries at
        their own positions, and the beacons are FPS(the earlier ones, fps_keep),
        all of them when there are no more than fps_keep; the picks are the
        head's trace. The prompt's keys and values go through append_kv."""
        assert all(not st.bq and not st.rq for st in self.heads), "prefill needs a fresh state"
        P = len(q_prompt[0])
        nr = min(self.n_rq, P)
        for h, st in enumerate(self.heads):
            rows = [np.asarray(r, dtype=np.uint16).copy() for r in q_prompt[h]]
            older = rows[:P - nr]
            if older:
                st.trace, keep = fps(bf16_to_f64(np.stack(older)), self.fps_keep)
                st.bq = [older[i] for i in keep]
            else:
                st.trace = []
            st.rq = deque((rows[P - nr + k], first_step + P - nr + k) for k in range(nr))

    def coverage(self, future_q) -> list[list[float]]:
        """Per query head, coverage() of its current observation set (beacons,
        then recents: what the next eviction scores) over future_q[h] rows."""
        return [coverage(list(st.bq) + [q for q, _ in st.rq], future_q[h])
                for h, st in enumerate(self.heads)]

    # -- state injection (steady-state samples for timing) -------------------
    def load_state(self, bq_rows, rq_rows, rq_pos, K, V, pos) -> None:
        """Set every head's beacons/recents and the cache slice directly."""
        for h, st in enumerate(self.heads):
            st.bq = [np.asarray(r, dtype=np.uint16).copy() for r in bq_rows[h]]
            st.rq = deque((np.asarray(r, dtype=np.uint16).copy(), int(p))
                          for r, p in zip(rq_rows[h], rq_pos))
        self.K = [np.asarray(r, dtype=np.uint16).copy() for r in K]
        self.V = [np.asarray(r, dtype=np.uint16).copy() for r in V]
        self.pos = [int(p) for p in pos]
