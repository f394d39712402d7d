"""Seeded synthetic decode stream: pre-RoPE queries, cached keys and values.

The structure follows what the BeaconKV pages describe about long reasoning
traces (reading notes, section 1 and Figures 1-4; rcap.io summary): most
queries are "local" and drift slowly, a sparse minority are "global" and
cluster tightly around a few directions in pre-RoPE space, and the earliest
keys (problem statement, plan) are the ones global queries revisit.

Recipe, per (layer, sequence, query head), at every decode step:
  * local  (probability 1 - global_frac): a random walk on the unit sphere,
    u <- normalize(u + walk_step * xi / sqrt(d)), xi ~ N(0, I);
  * global (probability global_frac): one of `centres` fixed unit directions of
    the query head's (layer, KV head), normalize(c + global_noise * xi / sqrt(d));
  * the direction is scaled by a lognormal(0, norm_sigma) norm.
Keys are drawn directly in cache space (the generator applies no rotation):
key j < aligned_keys is sqrt(d) * c_(j mod centres) + 0.1 * xi, later keys are
N(0, I). Values are N(0, I). Everything is rounded to bf16 (round to nearest
even) by torch's float32 -> bfloat16 conversion.

The stream runs on any torch device; CPU and CUDA draws differ, so a test
generates once and hands the same bytes to both the library and the oracle.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from .workloads import Workload


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (a copy, on the host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def _normalize(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


class SyntheticStream:
    """Generates step t's q_pre [layers][batch][heads][d] and k/v [layers][batch][kv_heads][d]."""

    def __init__(self, w: Workload, seed: int, device: str | torch.device = "cpu"):
        self.w = w
        self.device = torch.device(device)
        self.seed = int(seed)
        g = torch.Generator(device=self.device)
        g.manual_seed(self.seed)
        self._gq = g
        d = w.d
        self.centres = _normalize(torch.randn(w.layers, w.kv_heads, w.centres, d, generator=g,
                                              device=self.device))
        self.walk = _normalize(torch.randn(w.layers, w.batch, w.heads, d, generator=g,
                                           device=self.device))
        # query head h belongs to KV head h // group
        self._head_kv = torch.arange(w.heads, device=self.device) // w.group
        self.t = 0

    def queries(self) -> torch.Tensor:
        """Pre-RoPE queries of the next step (advances the stream by one step)."""
        w, g, d = self.w, self._gq, self.w.d
        shape = (w.layers, w.batch, w.heads)
        xi = torch.randn(*shape, d, generator=g, device=self.device)
        self.walk = _normalize(self.walk + w.walk_step * xi / math.sqrt(d))
        is_global = torch.rand(*shape, generator=g, device=self.device) < w.global_frac
        cidx = torch.randint(0, w.centres, shape, generator=g, device=self.device)
        noise = torch.randn(*shape, d, generator=g, device=self.device)
        lay = torch.arange(w.layers, device=self.device).view(-1, 1, 1).expand(shape)
        kvh = self._head_kv.view(1, 1, -1).expand(shape)
        cent = self.centres[lay, kvh, cidx]
        glob = _normalize(cent + w.global_noise * noise / math.sqrt(d))
        direction = torch.where(is_global.unsqueeze(-1), glob, self.walk)
        scale = torch.exp(w.norm_sigma * torch.randn(*shape, generator=g, device=self.device))
        self.t += 1
        return (direction * scale.unsqueeze(-1)).to(torch.bfloat16)

    def _kv_generator(self, pos: int, salt: int) -> torch.Generator:
        g = torch.Generator(device=self.device)
        g.manual_seed((self.seed * 1_000_003 + pos * 2 + salt) & 0x7FFF_FFFF_FFFF_FFFF)
        return g

    def keys_values(self, pos: int) -> tuple[torch.Tensor, torch.Tensor]:
        """Key and value written to the cache at absolute position `pos`."""
        w, d = self.w, self.w.d
        shape = (w.layers, w.batch, w.kv_heads, d)
        gk = self._kv_generator(pos, 0)
        k = torch.randn(*shape, generator=gk, device=self.device)
        if pos < w.aligned_keys:
            c = self.centres[:, :, pos % w.centres, :].unsqueeze(1)  # [L,1,Hkv,d]
            k = math.sqrt(d) * c + 0.1 * k
        gv = self._kv_generator(pos, 1)
        v = torch.randn(*shape, generator=gv, device=self.device)
        return k.to(torch.bfloat16), v.to(torch.bfloat16)

    def fill_cache(self, K: torch.Tensor, V: torch.Tensor, layer: int, rows: int) -> None:
        """Bulk-fill slots [0, rows) of one layer's [batch][kv_heads][max_cache][d] cache.

        A faster, different draw than keys_values(): used to set up large
        steady-state caches, where no step-by-step history is needed.
        """
        w, d = self.w, self.w.d
        g = self._kv_generator(1_000_000 + layer, 0)
        for b in range(w.batch):
            kb = torch.randn(w.kv_heads, rows, d, generator=g, device=self.device)
            na = min(rows, w.aligned_keys)
            idx = torch.arange(na, device=self.device) % w.centres
            kb[:, :na] = math.sqrt(d) * self.centres[layer][:, idx, :] + 0.1 * kb[:, :na]
            K[b, :, :rows].copy_(kb.to(torch.bfloat16))
            V[b, :, :rows].copy_(torch.randn(w.kv_heads, rows, d, generator=g,
                                             device=self.device).to(torch.bfloat16))
