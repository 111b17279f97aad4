"""Streaming quantized KV cache with an fp16 residual window (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it follows:
  * [explainer] 3.1 (grouped quantization with a residual): a prompt of l
    tokens is split into a part that is quantized in whole groups of G and a
    residual kept in fp16; when the residual has gathered R tokens they are
    quantized as a batch and the residual is emptied.
  * [axis-guide] "系统税收": per-channel key statistics span tokens that do
    not exist yet, so the newest tokens (up to R, e.g. 128) wait in a
    full-precision residual and are quantized once enough have gathered.
  * [explainer] 3.2 states the same residual mechanism for values; both keys
    and values flush together here (see the readings below).

Readings (where the pages are silent or disagree):
  * prefill split: the quantized prefix is Lq = G * ceil(max(l - R, 0) / G)
    tokens and the residual keeps r = l - Lq <= R tokens (a full residual of R
    tokens is allowed at rest);
  * the flush is lazy: an append that finds r == R first quantizes the R
    residual tokens (R/G key groups, R value tokens) at positions
    [Lq, Lq + R), then stores the new token as residual row 0;
  * group boundaries therefore always fall on multiples of G counted from
    token 0;
  * keys and values share one residual count and flush together (the
    one-token-at-a-time value queue of [explainer] 3.2 is OracleCacheFifo).

Parity status: pinned (streaming equals one-shot quantization of the same
token prefix; accounting invariants; residual holds the exact fp16 inputs).
"""
from __future__ import annotations

import numpy as np

from . import quant


def prefill_split(l: int, G: int, R: int):
    """(Lq, r): quantized-prefix length and residual length for an l-token prompt."""
    if l < 0:
        raise ValueError("negative length")
    over = max(l - R, 0)
    Lq = G * ((over + G - 1) // G)
    return Lq, l - Lq


class OracleCache:
    """Logical (unpacked) state of one KIVI cache: codes, steps, zeros, residual.

    Shapes ([B] batch, [H] kv heads, d head dim, Lq quantized tokens, r residual):
      k_codes uint8 [B][H][Lq][d], k_s / k_z fp16 [B][H][Lq/G][d]
      v_codes uint8 [B][H][Lq][d], v_s / v_z fp16 [B][H][Lq][d/G]
      k_res / v_res fp16 [B][H][r][d]
    """

    def __init__(self, B: int, H: int, d: int, bits: int, G: int, R: int):
        if R % G or R < G or d % G:
            raise ValueError("need R % G == 0, R >= G and d % G == 0")
        self.B, self.H, self.d, self.bits, self.G, self.R = B, H, d, bits, G, R
        self.k_codes = np.zeros((B, H, 0, d), np.uint8)
        self.k_s = np.zeros((B, H, 0, d), np.float16)
        self.k_z = np.zeros((B, H, 0, d), np.float16)
        self.v_codes = np.zeros((B, H, 0, d), np.uint8)
        self.v_s = np.zeros((B, H, 0, d // G), np.float16)
        self.v_z = np.zeros((B, H, 0, d // G), np.float16)
        self.k_res = np.zeros((B, H, 0, d), np.float16)
        self.v_res = np.zeros((B, H, 0, d), np.float16)
        self.flushes = 0

    @property
    def n_quant(self) -> int:
        return self.k_codes.shape[2]

    @property
    def n_resid(self) -> int:
        return self.k_res.shape[2]

    def _quantize_into(self, X_K, X_V):
        """Quantize whole groups of tokens and append them to the quantized part."""
        kc, ks, kz = quant.quantize_keys(X_K, self.bits, self.G)
        vc, vs, vz = quant.quantize_values(X_V, self.bits, self.G)
        cat = lambda a, b: np.concatenate([a, b], axis=2)
        self.k_codes, self.k_s, self.k_z = cat(self.k_codes, kc), cat(self.k_s, ks), cat(self.k_z, kz)
        self.v_codes, self.v_s, self.v_z = cat(self.v_codes, vc), cat(self.v_s, vs), cat(self.v_z, vz)

    def prefill(self, X_K: np.ndarray, X_V: np.ndarray):
        """Quantize the G-aligned prefix of a prompt and keep the tail in fp16."""
        if self.n_quant or self.n_resid:
            raise RuntimeError("prefill on a non-empty cache")
        l = X_K.shape[2]
        Lq, _ = prefill_split(l, self.G, self.R)
        if Lq:
            self._quantize_into(X_K[:, :, :Lq], X_V[:, :, :Lq])
        self.k_res = X_K[:, :, Lq:].copy()
        self.v_res = X_V[:, :, Lq:].copy()

    def append(self, k: np.ndarray, v: np.ndarray):
        """Add one token (k, v: fp16 [B][H][d]); flush first when the residual is full."""
        if self.n_resid == self.R:
            self._quantize_into(self.k_res, self.v_res)
            self.k_res = self.k_res[:, :, :0]
            self.v_res = self.v_res[:, :, :0]
            self.flushes += 1
        self.k_res = np.concatenate([self.k_res, k[:, :, None, :]], axis=2)
        self.v_res = np.concatenate([self.v_res, v[:, :, None, :]], axis=2)

    def keys_hat(self) -> np.ndarray:
        """All cached keys in fp64 [B][H][Lq + r][d]: dequantized prefix, then residual."""
        kq = quant.dequantize_keys(self.k_codes, self.k_s, self.k_z, self.G)
        return np.concatenate([kq, self.k_res.astype(np.float64)], axis=2)

    def values_hat(self) -> np.ndarray:
        """All cached values in fp64 [B][H][Lq + r][d]: dequantized prefix, then residual."""
        vq = quant.dequantize_values(self.v_codes, self.v_s, self.v_z, self.G)
        return np.concatenate([vq, self.v_res.astype(np.float64)], axis=2)


class OracleCacheFifo(OracleCache):
    """The same cache with the value residual kept as a queue ([explainer] 3.2).

    Keys behave exactly as in OracleCache (whole groups, flush of the R
    residual tokens when full).  Values follow [explainer] 3.2: new value
    tokens enter an fp16 queue; once it holds R tokens, the oldest token
    leaves the queue, is quantized on its own (per token, groups of G
    channels) and joins the quantized values; the newest R values stay fp16.

    Readings: after every call the queue holds the newest min(l, R) value
    tokens and the first max(l - R, 0) are quantized (an append pushes the
    new token and pops the oldest once the queue would exceed R; a prompt
    quantizes all but its last R values).  Because value groups lie within one
    token, the quantized values equal a one-shot per-token quantization of
    the same prefix.

    Extra state: v_codes / v_s / v_z cover the first max(l - R, 0) tokens
    (n_quant_v of them); v_res holds the queue in token order.

    Parity status: pinned (one-shot equality, the queue's contents, keys
    identical to OracleCache, hand-worked positions).
    """

    @property
    def n_quant_v(self) -> int:
        return self.v_codes.shape[2]

    def prefill(self, X_K: np.ndarray, X_V: np.ndarray):
        if self.n_quant or self.n_resid or self.n_quant_v or self.v_res.shape[2]:
            raise RuntimeError("prefill on a non-empty cache")
        l = X_K.shape[2]
        Lq, _ = prefill_split(l, self.G, self.R)
        if Lq:
            kc, ks, kz = quant.quantize_keys(X_K[:, :, :Lq], self.bits, self.G)
            self.k_codes, self.k_s, self.k_z = kc, ks, kz
        self.k_res = X_K[:, :, Lq:].copy()
        Lv = max(l - self.R, 0)
        if Lv:
            self.v_codes, self.v_s, self.v_z = quant.quantize_values(X_V[:, :, :Lv], self.bits, self.G)
        self.v_res = X_V[:, :, Lv:].copy()

    def append(self, k: np.ndarray, v: np.ndarray):
        # keys: as in OracleCache
        if self.n_resid == self.R:
            kc, ks, kz = quant.quantize_keys(self.k_res, self.bits, self.G)
            cat = lambda a, b: np.concatenate([a, b], axis=2)
            self.k_codes, self.k_s, self.k_z = cat(self.k_codes, kc), cat(self.k_s, ks), cat(self.k_z, kz)
            self.k_res = self.k_res[:, :, :0]
            self.flushes += 1
        self.k_res = np.concatenate([self.k_res, k[:, :, None, :]], axis=2)
        # values: push, then pop the oldest once the queue would exceed R
        self.v_res = np.concatenate([self.v_res, v[:, :, None, :]], axis=2)
        if self.v_res.shape[2] > self.R:
            vc, vs, vz = quant.quantize_values(self.v_res[:, :, :1], self.bits, self.G)
            cat = lambda a, b: np.concatenate([a, b], axis=2)
            self.v_codes, self.v_s, self.v_z = cat(self.v_codes, vc), cat(self.v_s, vs), cat(self.v_z, vz)
            self.v_res = self.v_res[:, :, 1:]

