"""CPU oracle for BeaconKV's periodic KV-cache eviction step.

TEST INFRASTRUCTURE. This package is the plain, slow, fp64 statement of what
the eviction step computes. It is imported only by the test suite, by
`__graft_entry__.smoke()` (to check one small GPU invocation) and by the
`cpu_baseline` / `--impl reference` legs of `bench.py`. The product path (the
CUDA library and its Python binding) never imports, calls or links it, and it
shares no code with that path.

Parity pins: every function is checked in tests/ against something other than
itself (closed forms, brute force, exact rational arithmetic, hand-derived
fixtures in tests/golden/). The score values themselves have no printed worked
example on the pages; they are pinned by invariants and special cases only
(softmax rows sum to one, the zero-beacon reduction to a separately written
SnapKV max formula, the single-row case).
"""

from .beaconkv import (
    bf16_to_f64,
    rope,
    exact_dot,
    gram_exact,
    cosine_matrix,
    coverage,
    fps,
    attention_weights,
    max_pool,
    mean_pool,
    select_keep,
    order_free_layout,
    UnitOracle,
)

__all__ = [
    "bf16_to_f64", "rope", "exact_dot", "gram_exact", "cosine_matrix", "coverage", "fps",
    "attention_weights", "max_pool", "mean_pool", "select_keep", "order_free_layout", "UnitOracle",
]
