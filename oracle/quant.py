"""Uniform asymmetric B-bit group quantization (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition followed ([axis-guide], "量化错误的真正组成", uniform integer
quantization): for one group of numbers, record the smallest as the zero
point; divide the group's range by the number of representable steps,
2^B - 1, to get the step size; round every element to the nearest step.
Consequences stated there, and pinned by the tests: every element's error is
at most half a step, and the step is range / (2^B - 1).

Readings where the pages leave a step open (each also listed in the design
notes):
  * arithmetic is IEEE fp32, round-to-nearest-even, one operation at a time
    (no fused multiply-add), on fp16 inputs;
  * the zero point and the step are stored as fp16; the step is rounded to
    fp16 BEFORE the codes are chosen, so codes are the nearest levels of the
    stored (dequantization) grid;
  * "round to the nearest step" ties go to the even code (rint);
  * a group whose stored step is 0 (all elements equal, or a range too small
    for fp16) gets all-zero codes and dequantizes to the zero point;
  * a signed zero as group minimum is stored as +0.

Grouping ([explainer] 3.1 pseudo-code, [axis-guide] keys / values sections,
[survey]): keys are quantized per channel over groups of G consecutive tokens
(the key tensor viewed as (-1, G, d)); values per token over groups of G
consecutive channels.

Parity status: pinned (hand-worked groups, half-step bound, level coverage,
brute-force nearest level, axis-isolation tests).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def levels(B: int) -> int:
    """Number of steps of a B-bit code, 2^B - 1 (the top code)."""
    return (1 << B) - 1


def quantize_groups(X: np.ndarray, B: int, axis: int):
    """Quantize fp16 array ``X`` with one group per slice along ``axis``.

    Returns ``(codes, s, z)``: codes uint8 with X's shape, and fp16 step ``s``
    and zero point ``z`` with ``axis`` reduced to length 1.
    """
    if X.dtype != np.float16:
        raise TypeError("inputs are fp16")
    L = F32(levels(B))
    x = X.astype(F32)                                   # exact widening
    # zero point: the group minimum ( +0 makes a -0 minimum canonical )
    mn = x.min(axis=axis, keepdims=True) + F32(0.0)
    mx = x.max(axis=axis, keepdims=True) + F32(0.0)
    z16 = mn.astype(np.float16)                         # exact: mn is an fp16 value
    # step: range / (2^B - 1) in fp32, then stored as fp16
    s16 = ((mx - mn) / L).astype(np.float16)
    s = s16.astype(F32)
    z = z16.astype(F32)
    # nearest level of the stored grid
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (x - z) / s
    ratio = np.where(s == F32(0.0), F32(0.0), ratio)
    codes = np.clip(np.rint(ratio), F32(0.0), L).astype(np.uint8)
    return codes, s16, z16


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """Dequantized value code*s + z, exactly, in fp64.

    The product and the sum are exact in fp64: every fp16 value is a multiple
    of 2^-24 below 2^16 and codes are below 2^8, so the result is a multiple of
    2^-24 below 2^25 (at most 49 significant bits).  This is the real number
    the stored (code, s, z) represent.
    """
    return codes.astype(np.float64) * s.astype(np.float64) + z.astype(np.float64)


def quantize_keys(X_K: np.ndarray, B: int, G: int):
    """Per-channel key quantization over groups of G tokens.

    ``X_K``: fp16 [..., l, d] with l a multiple of G.  Viewed as
    [..., l/G, G, d] and reduced over the G tokens of each group, so every
    (group, channel) pair gets its own step and zero point.
    Returns codes uint8 [..., l, d]; s, z fp16 [..., l/G, d].
    """
    *lead, l, d = X_K.shape
    if l % G:
        raise ValueError("key token count must be a multiple of G")
    Xg = X_K.reshape(*lead, l // G, G, d)
    codes, s, z = quantize_groups(Xg, B, axis=-2)
    return codes.reshape(*lead, l, d), s[..., 0, :], z[..., 0, :]


def quantize_values(X_V: np.ndarray, B: int, G: int):
    """Per-token value quantization over groups of G channels.

    ``X_V``: fp16 [..., l, d] with d a multiple of G.  Each token's channels
    are cut into d/G groups of G consecutive channels.
    Returns codes uint8 [..., l, d]; s, z fp16 [..., l, d/G].
    """
    *lead, l, d = X_V.shape
    if d % G:
        raise ValueError("head dim must be a multiple of G")
    Xg = X_V.reshape(*lead, l, d // G, G)
    codes, s, z = quantize_groups(Xg, B, axis=-1)
    return codes.reshape(*lead, l, d), s[..., 0], z[..., 0]


def dequantize_keys(codes, s, z, G: int) -> np.ndarray:
    """fp64 keys from per-channel codes: each group's (s, z) spread over its G tokens."""
    return dequantize(codes, np.repeat(s, G, axis=-2), np.repeat(z, G, axis=-2))


def dequantize_values(codes, s, z, G: int) -> np.ndarray:
    """fp64 values from per-token codes: each (s, z) spread over its G channels."""
    return dequantize(codes, np.repeat(s, G, axis=-1), np.repeat(z, G, axis=-1))
