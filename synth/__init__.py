"""Seeded synthetic inputs for the BeaconKV eviction step.

This package only draws random numbers and shapes them into queries, keys and
values. It holds none of the eviction method's arithmetic (no RoPE, no softmax,
no farthest-point sampling, no selection): both the CUDA library and the CPU
oracle consume the bf16 bytes it produces.
"""

from .workloads import WORKLOADS, Workload, kv_bytes_per_token
from .stream import SyntheticStream, to_bits

__all__ = ["WORKLOADS", "Workload", "kv_bytes_per_token", "SyntheticStream", "to_bits"]
