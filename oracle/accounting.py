"""Closed-form byte counts (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

  * fp16 KV-cache size ([explainer] 2.1): batch x sequence x 2 (K and V) x
    layers x hidden x sizeof(fp16).  [explainer] section 1 quotes about
    0.5 MB per token for LLaMA2-7B in fp16 (32 layers, hidden 4096).
  * quantized bytes per cached token and (batch, kv-head) slot: key and value
    codes (D*b/8 bytes each) plus their fp16 (step, zero) pairs - one pair per
    channel per G tokens for keys, one pair per G channels per token for
    values, i.e. 4*D/G bytes per token each.
  * algorithmic bytes of one decode call: every cached byte once (codes,
    steps, zeros, fp16 residual rows) plus the query and the output.

Parity status: pinned (LLaMA2-7B figure; per-token figures by hand).
"""
from __future__ import annotations


def fp16_kv_bytes(batch: int, seq: int, layers: int, hidden: int) -> int:
    return batch * seq * 2 * layers * hidden * 2


def quantized_bytes_per_token(D: int, b: int, G: int) -> int:
    return 2 * (D * b // 8) + 2 * (4 * D // G)


def decode_call_bytes(B: int, Hq: int, Hkv: int, D: int, b: int, G: int, Lq: int, r: int) -> int:
    cache = B * Hkv * (Lq * quantized_bytes_per_token(D, b, G) + r * 2 * D * 2)
    return cache + 2 * B * Hq * D * 2
