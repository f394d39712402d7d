"""BeaconKV periodic KV-cache eviction step for GB300 (sm_103a).

The work runs in hand-written CUDA kernels behind the C ABI of include/bkv.h
(libbkv.so, built in-tree by `build.build()`); `kv_cache_eviction_head_gb300.bkv`
is the ctypes binding with the same function names. There is no CPU fallback:
importing the binding without the built library raises ImportError.
"""

__all__ = ["build", "bkv"]
