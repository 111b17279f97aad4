"""Seeded synthetic inputs for the KIVI KV-cache path.

This module only draws random tensors with the shapes and value structure of
the workloads (keys with fixed outlier channels, an attention-sink token,
N(0,1) values and queries).  It holds none of the quantization or attention
arithmetic, so both the CPU oracle and the CUDA library can be fed from it.

Structure of the data (KV-cache axis-selection guide, unite.ai, section
"Keys: outliers sit in fixed channels"): a few key channels carry very large
magnitudes on every token, always the same channels; values show no channel
pattern; attention concentrates on a few "sink" tokens.

Synthetic recipe (per (batch, kv-head) slot):
  * K ~ N(0,1); ``n_out`` outlier channels are scaled by a per-channel factor
    on every token (prompt tokens and every appended token alike);
  * with ``sink=True`` a unit direction u is drawn per slot, K[token 0] is
    replaced by ``kappa * u`` and every decode query is
    ``0.5*sqrt(D)*u + N(0,1)`` so token 0 draws a large share of attention;
  * V ~ N(0,1); q ~ N(0,1) when there is no sink.
Everything is drawn in fp32 and rounded once to fp16 (round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class OutlierSpec:
    """How key outlier channels are drawn for each (batch, kv-head) slot.

    ``fixed``: exactly ``count`` channels, all scaled by ``scale_lo``.
    otherwise: count ~ U{count_lo..count_hi}, each scale ~ U[scale_lo, scale_hi].
    """
    count_lo: int = 2
    count_hi: int = 6
    scale_lo: float = 10.0
    scale_hi: float = 50.0
    fixed: bool = False


FIXED_4_X20 = OutlierSpec(count_lo=4, count_hi=4, scale_lo=20.0, scale_hi=20.0, fixed=True)
RANGE_2_6_X10_50 = OutlierSpec()


class SynthKV:
    """Deterministic generator of prompt K/V and per-step (q, k, v)."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 seed: int, outliers: OutlierSpec = RANGE_2_6_X10_50,
                 sink: bool = True, kappa: float = 40.0, device="cpu"):
        if n_q_heads % n_kv_heads:
            raise ValueError("n_q_heads must be a multiple of n_kv_heads")
        self.B, self.Hq, self.Hkv, self.D = batch, n_q_heads, n_kv_heads, head_dim
        self.seed, self.sink, self.kappa = seed, sink, kappa
        self.device = torch.device(device)
        g = torch.Generator(device="cpu").manual_seed(seed)
        # per-channel key scale: 1 for ordinary channels, the outlier factor otherwise
        scale = torch.ones(batch, n_kv_heads, head_dim, dtype=torch.float32)
        for b in range(batch):
            for h in range(n_kv_heads):
                if outliers.fixed:
                    n = outliers.count_lo
                else:
                    n = int(torch.randint(outliers.count_lo, outliers.count_hi + 1, (1,), generator=g))
                ch = torch.randperm(head_dim, generator=g)[:n]
                f = outliers.scale_lo + (outliers.scale_hi - outliers.scale_lo) * torch.rand(n, generator=g)
                scale[b, h, ch] = f
        self.key_scale = scale.to(self.device)
        u = torch.randn(batch, n_kv_heads, head_dim, generator=g, dtype=torch.float32)
        self.sink_dir = (u / u.norm(dim=-1, keepdim=True)).to(self.device)

    # -- helpers -------------------------------------------------------------
    def _gen(self, tag: int) -> torch.Generator:
        gen = torch.Generator(device=self.device)
        gen.manual_seed((self.seed * 1_000_003 + tag) % (2**63 - 1))
        return gen

    def _normal(self, shape, gen) -> torch.Tensor:
        return torch.randn(*shape, generator=gen, dtype=torch.float32, device=self.device)

    # -- prompt ---------------------------------------------------------------
    def prompt(self, length: int):
        """Prompt keys and values, fp16, layout [B][Hkv][length][D]."""
        B, H, D = self.B, self.Hkv, self.D
        gk, gv = self._gen(1), self._gen(2)
        K = torch.empty(B, H, length, D, dtype=torch.float16, device=self.device)
        V = torch.empty_like(K)
        for b in range(B):  # per batch row to bound the fp32 temporaries
            kb = self._normal((H, length, D), gk) * self.key_scale[b][:, None, :]
            if self.sink and length > 0:
                kb[:, 0, :] = self.kappa * self.sink_dir[b]
            K[b] = kb.to(torch.float16)
            V[b] = self._normal((H, length, D), gv).to(torch.float16)
        return K, V

    # -- one decode step -------------------------------------------------------
    def step(self, s: int):
        """(q [B][Hq][D], k [B][Hkv][D], v [B][Hkv][D]) for decode step ``s``, fp16."""
        B, Hq, Hkv, D = self.B, self.Hq, self.Hkv, self.D
        gen = self._gen(1000 + 3 * s)
        q = self._normal((B, Hq, D), gen)
        if self.sink:
            kv_of = torch.arange(Hq, device=self.device) // (Hq // Hkv)
            q = q + 0.5 * math.sqrt(D) * self.sink_dir[:, kv_of, :]
        k = self._normal((B, Hkv, D), gen) * self.key_scale
        v = self._normal((B, Hkv, D), gen)
        return q.to(torch.float16), k.to(torch.float16), v.to(torch.float16)
