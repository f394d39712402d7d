"""The bounds-checked build (libbkv_checked.so, -DBKV_CHECKED) on the tiny
parity cases. In that build every computed slot, row and offset the kernels
index with (keep-set writes, compaction sources and destinations, order-free
holes, FPS picks) is tested before use; a failed test latches
BKV_ERR_INTERNAL, which bkv_sync raises. The cases run in a child process
that loads the checked library (BKV_LIBRARY=checked) and must all match the
oracle with no latched status."""

from __future__ import annotations

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent('''
    from synth import WORKLOADS
    from tests.lockstep import run_lockstep
    from kv_cache_eviction_head_gb300 import bkv
    assert bkv.library_path().endswith("libbkv_checked.so"), bkv.library_path()
    T = WORKLOADS["tiny"]
    cases = [
        ("tiny_stream", T, {}),
        ("order_free", T, dict(order_free=True)),
        ("radix_drops", T.with_(budget=160, period=48, steps=520), {}),
        ("radix_drops_order_free", T.with_(budget=160, period=48, steps=520), dict(order_free=True)),
        ("period_one", T.with_(period=1, steps=200), {}),
        ("odd_drops", T.with_(period=17, steps=260), {}),
        ("row_chunks_gqa12", T.with_(heads=12, kv_heads=1, steps=240), {}),
        ("gqa7_mean", T.with_(heads=7, kv_heads=1, steps=240), dict(pool="mean")),
        ("batch_layers", T.with_(layers=2, batch=3, heads=8, kv_heads=2, steps=200), {}),
        ("prefill_144", T.with_(steps=320), dict(prefill=144)),
        ("many_tiles", T.with_(budget=1000, steps=1100, heads=8, kv_heads=2), {}),
    ]
    for i, (name, w, kw) in enumerate(cases):
        rep = run_lockstep(w, seed=0xC4EC0 + i, **kw)
        assert not rep.failures, (name, rep.failures[:3])
        assert rep.evictions >= 1 and rep.units_checked >= rep.evictions, name
        print(name, rep.evictions, rep.units_checked, flush=True)
    print("CHECKED_OK")
''')


def test_checked_build_runs_the_tiny_parity_cases_clean():
    from kv_cache_eviction_head_gb300.build import build
    build(checked=True)
    env = {**os.environ, "BKV_LIBRARY": "checked"}
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0 and "CHECKED_OK" in r.stdout, (r.stdout[-3000:] + r.stderr[-3000:])
