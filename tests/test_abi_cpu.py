"""Host-only checks of the C ABI: the library builds, loads and exports every
entry point include/bkv.h declares, and the size/validation logic that runs
before any CUDA call returns the documented codes. Nothing here touches a GPU."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bkv():
    from kv_cache_eviction_head_gb300.build import build
    build()
    from kv_cache_eviction_head_gb300 import bkv as mod
    return mod


def declared_functions():
    with open(os.path.join(ROOT, "include", "bkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bkv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_documented_api():
    names = declared_functions()
    for n in ["bkv_workspace_bytes", "bkv_create", "bkv_append_queries", "bkv_evict", "bkv_sync",
              "bkv_get_fps_trace", "bkv_destroy", "bkv_status_str"]:
        assert n in names


def test_library_exports_every_declared_symbol(bkv):
    lib = ctypes.CDLL(bkv.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(bkv.EXPORTED) == declared_functions()


def cfg_for(bkv, **over):
    base = dict(heads=32, kv_heads=8, d=128, budget=2048, period=16, prefix=4, recent=16,
                fps_cap=32, fps_keep=16, layers=36, batch=192, max_cache=2064, rope_theta=1e6)
    base.update(over)
    return bkv.make_config(**base)


def test_workspace_bytes_matches_the_layout(bkv):
    c = cfg_for(bkv)
    heads = 36 * 192 * 32
    n_rq = 16
    want = 256 + 256 * ((1 + n_rq) * 64 * 8 // 256) + heads * 32 * 256 + heads * n_rq * 256 \
        + ((heads * 16 + 255) // 256) * 256
    assert bkv.bkv_workspace_bytes(c) == want
    c2 = cfg_for(bkv, flags=bkv.BKV_FLAG_KEEP_SCORES)
    assert bkv.bkv_workspace_bytes(c2) == want + 36 * 192 * 8 * 2064 * 4
    c3 = cfg_for(bkv, flags=bkv.BKV_FLAG_ORDER_FREE)   # the compaction layout needs no state
    assert bkv.bkv_workspace_bytes(c3) == want


@pytest.mark.parametrize("over,code", [
    (dict(heads=30), 1), (dict(kv_heads=0), 1), (dict(budget=0), 1), (dict(period=0), 1),
    (dict(prefix=2000, recent=100), 1), (dict(fps_keep=32), 1), (dict(fps_keep=-1), 1),
    (dict(max_cache=2048), 1), (dict(rope_theta=0.0), 1), (dict(flags=8), 1),
    (dict(d=64), 7), (dict(fps_cap=40, fps_keep=16), 7), (dict(layers=129), 7),
])
def test_invalid_configs_return_documented_codes(bkv, over, code):
    with pytest.raises(bkv.BkvError) as ei:
        bkv.bkv_workspace_bytes(cfg_for(bkv, **over))
    assert ei.value.code == code


def test_create_rejects_bad_workspace_before_any_cuda_call(bkv):
    c = cfg_for(bkv, layers=1, batch=1)
    need = bkv.bkv_workspace_bytes(c)
    out = ctypes.c_void_p(0)
    st = bkv.raw_status("bkv_create", ctypes.byref(c), None, ctypes.c_size_t(need), None, ctypes.byref(out))
    assert st == bkv.BKV_ERR_WORKSPACE and not out.value
    st = bkv.raw_status("bkv_create", ctypes.byref(c), ctypes.c_void_p(4096 * 1024),
                        ctypes.c_size_t(need - 1), None, ctypes.byref(out))
    assert st == bkv.BKV_ERR_WORKSPACE
    st = bkv.raw_status("bkv_create", ctypes.byref(c), ctypes.c_void_p(4096 * 1024 + 16),
                        ctypes.c_size_t(need), None, ctypes.byref(out))
    assert st == bkv.BKV_ERR_WORKSPACE


def test_null_handle_calls_are_rejected(bkv):
    for name, args in [("bkv_append_queries", (None, None, 0)), ("bkv_sync", (None,)),
                       ("bkv_evict", (None, None, None, 0, 0, None)),
                       ("bkv_get_fps_trace", (None, None, 0)), ("bkv_set_stream", (None, None)),
                       ("bkv_selftest_wait", (None, 1000))]:
        assert bkv.raw_status(name, *args) == bkv.BKV_ERR_INVALID_ARG


def test_status_strings(bkv):
    assert bkv.bkv_status_str(0) == "BKV_OK"
    assert bkv.bkv_status_str(5) == "BKV_ERR_NONFINITE"
    assert bkv.bkv_status_str(99) == "BKV_ERR_UNKNOWN"


@pytest.mark.parametrize("over,beacons,recents,cache_len,status,code", [
    (dict(), 16, 16, 2064, 0, 0),            # valid: would launch, not run here
    (dict(), 16, 17, 2064, 0, 1),            # more recents than the ring holds
    (dict(fps_keep=0), 0, 33, 2064, 0, 1),   # beyond the 32 recents of the static table
    (dict(), 32, 0, 2064, 0, 1),             # beacons == fps_cap
    (dict(), 0, 0, 2064, 0, 1),              # no observation row at all
    (dict(), -1, 16, 2064, 0, 1),
    (dict(flags=8), 16, 16, 2064, 0, 1),     # unknown flag
    (dict(), 16, 16, 2048, 0, 1),            # cache_len not above the budget
    (dict(), 16, 16, 2065, 0, 1),            # cache_len beyond max_cache
    (dict(), 16, 16, 2064, 4096 + 2, 1),     # misaligned status word
    (dict(d=64), 16, 16, 2064, 0, 7),
    (dict(layers=129), 16, 16, 2064, 0, 7),
])
def test_noalloc_argument_checks_before_any_cuda_call(bkv, over, beacons, recents, cache_len, status, code):
    """bkv_score_select_noalloc validates everything on the host and returns
    the documented code before it touches the device (fake, aligned device
    addresses are enough: nothing is dereferenced)."""
    c = cfg_for(bkv, **{"layers": 2, "batch": 1, **over})
    K = (ctypes.c_void_p * max(c.layers, 1))(*[4096 * (i + 1) for i in range(max(c.layers, 1))])
    args = (ctypes.byref(c), ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), beacons, recents, K,
            cache_len, 5000, ctypes.c_void_p(3 << 20), ctypes.c_void_p(status), None)
    if code == 0:
        return  # the valid call would launch kernels: covered by the GPU tests
    assert bkv.raw_status("bkv_score_select_noalloc", *args) == code
