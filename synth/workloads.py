"""Workload shapes for the eviction step.

Each workload is a model head shape (layers, query heads, KV heads, head dim,
RoPE base) plus the eviction schedule (budget, period, prefix, recent window,
query-buffer bounds) and the synthetic stream that drives it. The head shapes
follow the models the BeaconKV pages evaluate (Qwen3-4B, Qwen3-14B,
R1-Distill-Qwen-7B; BeaconKV reading notes, section 3.1); the 16+16
beacon/recent split and the 32 -> 16 buffer follow the same notes, section 2.2
(eq. 9) and Table 1.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    heads: int
    kv_heads: int
    d: int
    theta: float
    budget: int
    period: int
    prefix: int
    recent: int
    fps_cap: int
    fps_keep: int
    centres: int          # cluster centres of the "global" queries, per (layer, KV head)
    steps: int            # decode steps in the synthetic stream
    global_frac: float = 0.1
    walk_step: float = 0.05
    global_noise: float = 0.1
    norm_sigma: float = 0.25
    aligned_keys: int = 64
    cache_slots: int = 0  # cache capacity when a prompt may exceed budget + period (0: budget + period)

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    @property
    def max_cache(self) -> int:
        return max(self.cache_slots, self.budget + self.period)

    @property
    def units(self) -> int:
        """Independent eviction units: (sequence, layer, KV head)."""
        return self.layers * self.batch * self.kv_heads

    @property
    def evictions_per_round(self) -> int:
        """One eviction = one (layer, sequence) pair."""
        return self.layers * self.batch

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def kv_bytes_per_token(layers: int, kv_heads: int, d: int, elem_bytes: int = 2) -> int:
    """Bytes of K plus V that one token adds to the cache across all layers."""
    return layers * kv_heads * d * 2 * elem_bytes


_COMMON = dict(d=128, period=16, prefix=4, recent=16, fps_cap=32, fps_keep=16)

WORKLOADS: dict[str, Workload] = {
    # Small case the oracle finishes in seconds: one unit, a 512-step stream.
    "tiny": Workload(name="tiny", layers=1, batch=1, heads=4, kv_heads=1, theta=1e6,
                     budget=128, centres=6, steps=512, **_COMMON),
    # Qwen3-4B head shape, batch 1: one eviction over all layers.
    "qwen3_4b_b1": Workload(name="qwen3_4b_b1", layers=36, batch=1, heads=32, kv_heads=8,
                            theta=1e6, budget=2048, centres=6, steps=2064, **_COMMON),
    # Qwen3-4B head shape at the matched-budget batch of 192 (BeaconKV notes, Table 4).
    "qwen3_4b_b192": Workload(name="qwen3_4b_b192", layers=36, batch=192, heads=32, kv_heads=8,
                              theta=1e6, budget=2048, centres=6, steps=4096, **_COMMON),
    # Qwen3-14B head shape, batch 64, 1K budget, 8 centres per head.
    "qwen3_14b_b64": Workload(name="qwen3_14b_b64", layers=40, batch=64, heads=40, kv_heads=8,
                              theta=1e6, budget=1024, centres=8, steps=4096, **_COMMON),
}

# R1-Distill-Qwen-7B head shape, batch 128, budget sweep.
for _b in (256, 512, 1024, 2048, 4096):
    WORKLOADS[f"r1_qwen7b_b128_k{_b}"] = Workload(
        name=f"r1_qwen7b_b128_k{_b}", layers=28, batch=128, heads=28, kv_heads=4, theta=1e4,
        budget=_b, centres=6, steps=32768, **_COMMON)

# The pages' eviction schedule (BeaconKV reading notes §2.3): the cache grows to
# B_max = 2048 and is cut to B_min = 7/8 B_max = 1792, so each eviction drops
# 256 slots and 256 decode steps separate evictions (FPS still runs whenever
# the beacon buffer fills, every 16 appends). Qwen3-4B head shape, batch 192.
WORKLOADS["qwen3_4b_b192_sched78"] = WORKLOADS["qwen3_4b_b192"].with_(
    name="qwen3_4b_b192_sched78", budget=1792, period=256)

