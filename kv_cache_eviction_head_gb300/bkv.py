"""Thin ctypes binding of libbkv (include/bkv.h), same names as the C ABI.

Argument marshalling only: tensors become device pointers, a torch stream
becomes its cudaStream_t, status codes become exceptions. Every step of the
eviction runs in the library's CUDA kernels. The library must be built
(`kv_cache_eviction_head_gb300.build.build()`); importing this module without
it raises ImportError.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

# BKV_LIBRARY=checked loads the bounds-checked build (libbkv_checked.so)
_VARIANTS = {"": "libbkv.so", "checked": "libbkv_checked.so"}
_variant = os.environ.get("BKV_LIBRARY", "")
if _variant not in _VARIANTS:
    raise ImportError(f"BKV_LIBRARY={_variant!r}: expected one of {sorted(_VARIANTS)}")
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _VARIANTS[_variant])
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with kv_cache_eviction_head_gb300.build.build()"
                      + (" (checked=True)" if _variant else ""))
_lib = ctypes.CDLL(_LIB_PATH)

BKV_OK = 0
BKV_ERR_INVALID_ARG = 1
BKV_ERR_STATE = 2
BKV_ERR_WORKSPACE = 3
BKV_ERR_CUDA = 4
BKV_ERR_NONFINITE = 5
BKV_ERR_TIMEOUT = 6
BKV_ERR_UNSUPPORTED = 7
BKV_ERR_INTERNAL = 8
BKV_FLAG_KEEP_SCORES = 1
BKV_FLAG_ORDER_FREE = 2
BKV_FLAG_MEAN_POOL = 4

EXPORTED = ["bkv_workspace_bytes", "bkv_create", "bkv_set_stream", "bkv_append_queries",
            "bkv_evict", "bkv_prefill", "bkv_coverage", "bkv_selftest_wait", "bkv_sync",
            "bkv_get_fps_trace", "bkv_get_scores", "bkv_get_head_state",
            "bkv_profile", "bkv_profile_read", "bkv_score_select_noalloc", "bkv_get_stats",
            "bkv_destroy", "bkv_status_str"]
KERNELS = ["append", "rope", "score_select", "fps", "coverage", "prefill"]


class BkvConfig(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("d", ctypes.c_int32),
                ("budget", ctypes.c_int32), ("period", ctypes.c_int32), ("prefix", ctypes.c_int32),
                ("recent", ctypes.c_int32), ("fps_cap", ctypes.c_int32), ("fps_keep", ctypes.c_int32),
                ("layers", ctypes.c_int32), ("batch", ctypes.c_int32), ("max_cache", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("flags", ctypes.c_int32)]


class BkvStats(ctypes.Structure):
    _fields_ = [("evictions", ctypes.c_uint64), ("fps_calls", ctypes.c_uint64),
                ("rows_moved", ctypes.c_uint64), ("beacons", ctypes.c_int32),
                ("recents", ctypes.c_int32), ("cache_len", ctypes.c_int32),
                ("last_step", ctypes.c_int64)]


class BkvKernelTimes(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 6), ("launches", ctypes.c_uint64 * 6)]


_vp, _sz, _i32, _i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
_lib.bkv_workspace_bytes.argtypes = [ctypes.POINTER(BkvConfig), ctypes.POINTER(_sz)]
_lib.bkv_create.argtypes = [ctypes.POINTER(BkvConfig), _vp, _sz, _vp, ctypes.POINTER(_vp)]
_lib.bkv_set_stream.argtypes = [_vp, _vp]
_lib.bkv_append_queries.argtypes = [_vp, _vp, _i64]
_lib.bkv_evict.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _i64, _vp]
_lib.bkv_coverage.argtypes = [_vp, _vp, _i32, _vp]
_lib.bkv_prefill.argtypes = [_vp, _vp, _i32, _i64, _vp]
_lib.bkv_sync.argtypes = [_vp]
_lib.bkv_selftest_wait.argtypes = [_vp, _i64]
_lib.bkv_get_fps_trace.argtypes = [_vp, _vp, _sz]
_lib.bkv_get_scores.argtypes = [_vp, _vp, _sz]
_lib.bkv_get_head_state.argtypes = [_vp, _i32, _i32, _i32, _vp, _sz]
_lib.bkv_get_stats.argtypes = [_vp, ctypes.POINTER(BkvStats)]
_lib.bkv_profile.argtypes = [_vp, _i32]
_lib.bkv_profile_read.argtypes = [_vp, ctypes.POINTER(BkvKernelTimes)]
_lib.bkv_score_select_noalloc.argtypes = [ctypes.POINTER(BkvConfig), _vp, _vp, _i32, _i32,
                                          ctypes.POINTER(_vp), _i32, _i64, _vp, _vp, _vp]
_lib.bkv_destroy.argtypes = [_vp]
_lib.bkv_destroy.restype = None
_lib.bkv_status_str.argtypes = [_i32]
_lib.bkv_status_str.restype = ctypes.c_char_p
for _n in EXPORTED[:-2]:
    getattr(_lib, _n).restype = ctypes.c_int


class BkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {bkv_status_str(code)}")


def bkv_status_str(code: int) -> str:
    return _lib.bkv_status_str(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != BKV_OK:
        raise BkvError(code, where)


def _check_tensor(t, name: str, dtype, shape) -> None:
    """Raises ValueError unless t is a contiguous CUDA tensor of this dtype and shape."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}"
                         f"{'' if t.is_contiguous() else ' (not contiguous)'}")


def _check_layers(ts, name: str, cfg) -> None:
    """`layers` bf16 caches [batch][kv_heads][max_cache][d], one per layer."""
    import torch
    if len(ts) != cfg.layers:
        raise ValueError(f"{name}: expected {cfg.layers} per-layer tensors, got {len(ts)}")
    for l, t in enumerate(ts):
        _check_tensor(t, f"{name}[{l}]", torch.bfloat16, (cfg.batch, cfg.kv_heads, cfg.max_cache, cfg.d))


def _stream_ptr(stream) -> int:
    if stream is None:
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def make_config(*, heads, kv_heads, d, budget, period, prefix, recent, fps_cap=32, fps_keep=16,
                layers, batch, max_cache, rope_theta, flags=0) -> BkvConfig:
    return BkvConfig(heads, kv_heads, d, budget, period, prefix, recent, fps_cap, fps_keep, layers,
                     batch, max_cache, float(rope_theta), flags)


def bkv_workspace_bytes(cfg: BkvConfig) -> int:
    n = _sz(0)
    _check(_lib.bkv_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "bkv_workspace_bytes")
    return n.value


@dataclass
class Handle:
    ptr: int
    cfg: BkvConfig
    workspace: object  # keeps the caller's workspace tensor alive


def bkv_create(cfg: BkvConfig, workspace, stream=None) -> Handle:
    """workspace: a uint8 CUDA tensor of at least bkv_workspace_bytes(cfg) bytes."""
    out = _vp(0)
    _check(_lib.bkv_create(ctypes.byref(cfg), _vp(workspace.data_ptr()), _sz(workspace.numel() * workspace.element_size()),
                           _vp(_stream_ptr(stream)), ctypes.byref(out)), "bkv_create")
    return Handle(out.value, cfg, workspace)


def bkv_set_stream(h: Handle, stream) -> None:
    _check(_lib.bkv_set_stream(_vp(h.ptr), _vp(_stream_ptr(stream))), "bkv_set_stream")


def bkv_append_queries(h: Handle, q_pre, step: int) -> None:
    """q_pre: bf16 CUDA tensor [layers][batch][heads][d], contiguous."""
    import torch
    c = h.cfg
    _check_tensor(q_pre, "q_pre", torch.bfloat16, (c.layers, c.batch, c.heads, c.d))
    _check(_lib.bkv_append_queries(_vp(h.ptr), _vp(q_pre.data_ptr()), _i64(step)), "bkv_append_queries")


def bkv_evict(h: Handle, K, V, cache_len: int, step: int, kept) -> None:
    """K, V: sequences of `layers` bf16 CUDA tensors [batch][kv_heads][max_cache][d];
    kept: int32 CUDA tensor [layers][batch][kv_heads][budget]."""
    import torch
    c = h.cfg
    _check_layers(K, "K", c)
    _check_layers(V, "V", c)
    _check_tensor(kept, "kept", torch.int32, (c.layers, c.batch, c.kv_heads, c.budget))
    n = len(K)
    kp = (_vp * n)(*[t.data_ptr() for t in K])
    vp = (_vp * n)(*[t.data_ptr() for t in V])
    _check(_lib.bkv_evict(_vp(h.ptr), kp, vp, _i32(cache_len), _i64(step), _vp(kept.data_ptr())),
           "bkv_evict")


def bkv_evict_ptrs(h: Handle, kptrs, vptrs, cache_len: int, step: int, kept_ptr: int) -> None:
    """bkv_evict with raw device pointers (pre-marshalled pointer arrays allowed)."""
    _check(_lib.bkv_evict(_vp(h.ptr), kptrs, vptrs, _i32(cache_len), _i64(step), _vp(kept_ptr)),
           "bkv_evict")


def bkv_prefill(h: Handle, q_prompt, first_step: int, trace_out=None) -> None:
    """q_prompt: bf16 CUDA tensor [P][layers][batch][heads][d]; trace_out: optional
    int32 CUDA tensor [layers][batch][heads][min(fps_keep, P - recents)]."""
    import torch
    c = h.cfg
    P = q_prompt.shape[0] if q_prompt.dim() == 5 else -1
    _check_tensor(q_prompt, "q_prompt", torch.bfloat16, (P, c.layers, c.batch, c.heads, c.d))
    if trace_out is not None:
        n_rq = c.fps_cap - c.fps_keep
        m = min(c.fps_keep, P - min(n_rq, P))
        _check_tensor(trace_out, "trace_out", torch.int32, (c.layers, c.batch, c.heads, m))
    _check(_lib.bkv_prefill(_vp(h.ptr), _vp(q_prompt.data_ptr()), _i32(q_prompt.shape[0]),
                            _i64(first_step), _vp(trace_out.data_ptr() if trace_out is not None else 0)),
           "bkv_prefill")


def bkv_coverage(h: Handle, q_future, out) -> None:
    """q_future: bf16 CUDA tensor [n_future][layers][batch][heads][d];
    out: float64 CUDA tensor [layers][batch][heads][n_future]."""
    import torch
    c = h.cfg
    n = q_future.shape[0] if q_future.dim() == 5 else -1
    _check_tensor(q_future, "q_future", torch.bfloat16, (n, c.layers, c.batch, c.heads, c.d))
    _check_tensor(out, "out", torch.float64, (c.layers, c.batch, c.heads, n))
    _check(_lib.bkv_coverage(_vp(h.ptr), _vp(q_future.data_ptr()), _i32(q_future.shape[0]),
                             _vp(out.data_ptr())), "bkv_coverage")


def bkv_sync(h: Handle) -> None:
    _check(_lib.bkv_sync(_vp(h.ptr)), "bkv_sync")


def bkv_selftest_wait(h: Handle, wait_cycles: int) -> None:
    """Enqueues the bounded-wait self-test; the next bkv_sync raises BKV_ERR_TIMEOUT."""
    _check(_lib.bkv_selftest_wait(_vp(h.ptr), _i64(wait_cycles)), "bkv_selftest_wait")


def bkv_get_fps_trace(h: Handle) -> np.ndarray:
    c = h.cfg
    out = np.empty((c.layers, c.batch, c.heads, c.fps_keep), dtype=np.int8)
    _check(_lib.bkv_get_fps_trace(_vp(h.ptr), _vp(out.ctypes.data), _sz(out.nbytes)), "bkv_get_fps_trace")
    return out


def bkv_get_scores(h: Handle) -> np.ndarray:
    c = h.cfg
    out = np.empty((c.layers, c.batch, c.kv_heads, c.max_cache), dtype=np.float32)
    _check(_lib.bkv_get_scores(_vp(h.ptr), _vp(out.ctypes.data), _sz(out.size)), "bkv_get_scores")
    return out


def bkv_get_head_state(h: Handle, layer: int, seq: int, head: int) -> np.ndarray:
    """uint16 [fps_cap + n_rq][d]: beacon rows, then the recent ring slots."""
    c = h.cfg
    out = np.empty((c.fps_cap + c.fps_cap - c.fps_keep, c.d), dtype=np.uint16)
    _check(_lib.bkv_get_head_state(_vp(h.ptr), layer, seq, head, _vp(out.ctypes.data), _sz(out.size)),
           "bkv_get_head_state")
    return out


def bkv_profile(h: Handle, enable: bool) -> None:
    _check(_lib.bkv_profile(_vp(h.ptr), _i32(1 if enable else 0)), "bkv_profile")


def bkv_profile_read(h: Handle) -> dict:
    """{kernel name: (summed ms, launches)} since profiling was enabled."""
    t = BkvKernelTimes()
    _check(_lib.bkv_profile_read(_vp(h.ptr), ctypes.byref(t)), "bkv_profile_read")
    return {k: (t.ms[i], int(t.launches[i])) for i, k in enumerate(KERNELS)}


def bkv_score_select_noalloc(cfg: BkvConfig, bq, rq, beacons: int, recents: int, K,
                             cache_len: int, step: int, kept, status=None, stream=None) -> None:
    """Score + keep-set selection without a handle or workspace (see include/bkv.h).
    bq: bf16 CUDA tensor [layers][batch][heads][fps_cap][d]; rq: bf16 CUDA tensor
    [layers][batch][heads][fps_cap - fps_keep][d]; K: `layers` bf16 CUDA tensors
    [batch][kv_heads][max_cache][d]; kept: int32 CUDA tensor
    [layers][batch][kv_heads][budget]; status: optional uint32-sized CUDA tensor
    (int32, one element) receiving the device-side status."""
    import torch
    c = cfg
    n_rq = c.fps_cap - c.fps_keep
    _check_tensor(bq, "bq", torch.bfloat16, (c.layers, c.batch, c.heads, c.fps_cap, c.d))
    _check_tensor(rq, "rq", torch.bfloat16, (c.layers, c.batch, c.heads, n_rq, c.d))
    _check_layers(K, "K", c)
    _check_tensor(kept, "kept", torch.int32, (c.layers, c.batch, c.kv_heads, c.budget))
    if status is not None:
        _check_tensor(status, "status", torch.int32, (1,))
    n = len(K)
    kp = (_vp * n)(*[t.data_ptr() for t in K])
    _check(_lib.bkv_score_select_noalloc(ctypes.byref(cfg), _vp(bq.data_ptr()), _vp(rq.data_ptr()),
                                         _i32(beacons), _i32(recents), kp, _i32(cache_len),
                                         _i64(step), _vp(kept.data_ptr()),
                                         _vp(status.data_ptr() if status is not None else 0),
                                         _vp(_stream_ptr(stream))),
           "bkv_score_select_noalloc")


def bkv_get_stats(h: Handle) -> BkvStats:
    s = BkvStats()
    _check(_lib.bkv_get_stats(_vp(h.ptr), ctypes.byref(s)), "bkv_get_stats")
    return s


def bkv_destroy(h: Handle) -> None:
    if h.ptr:
        _lib.bkv_destroy(_vp(h.ptr))
        h.ptr = 0


def raw_status(fn_name: str, *args) -> int:
    """Calls a C entry point and returns its status code (tests of the error paths)."""
    return getattr(_lib, fn_name)(*args)


def library_path() -> str:
    return _LIB_PATH
