"""Single-query decode attention over the cached keys and values (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it follows ([axis-guide], "为什么 KV 缓存是问题所在" and "值：直觉在哪里
破裂"): at every generated token the whole KV cache is read; the attention
output is the sum of the value vectors over tokens weighted by the softmax
attention scores of the query against the keys.

Readings: the score scale is 1/sqrt(d) unless a scale is given; there is no
mask (one new query attends to every cached token, the newest one included);
query head h reads kv head h // (Hq / Hkv).  Everything is fp64: the logits
are softmax(scale * q . k_t), taken after subtracting the maximum logit.

Parity status: pinned (uniform weights give the mean, two-token closed form,
dominant-token bound, permutation and logit-shift invariance, grouped-query
equals replicated heads).
"""
from __future__ import annotations

import math

import numpy as np


def decode_attention(q: np.ndarray, K_hat: np.ndarray, V_hat: np.ndarray,
                     scale: float | None = None):
    """o[b, h] = sum_t softmax_t(scale * q[b,h] . K_hat[b,kv,t]) * V_hat[b,kv,t].

    q: [B][Hq][d] (any float dtype, used exactly in fp64);
    K_hat, V_hat: fp64 [B][Hkv][T][d] with T >= 1.
    Returns (o fp64 [B][Hq][d], lse fp64 [B][Hq]) where lse is the natural-log
    sum of exp of the scaled logits.
    """
    B, Hq, d = q.shape
    _, Hkv, T, _ = K_hat.shape
    if T < 1:
        raise ValueError("attention over an empty cache")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rep = Hq // Hkv
    qd = q.astype(np.float64)
    o = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // rep
            logits = scale * (K_hat[b, kv] * qd[b, h][None, :]).sum(axis=1)
            m = logits.max()
            e = np.exp(logits - m)
            l = e.sum()
            o[b, h] = (e[:, None] * V_hat[b, kv]).sum(axis=0) / l
            lse[b, h] = m + math.log(l)
    return o, lse
