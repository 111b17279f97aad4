"""Pins for the oracle's group quantizer (no GPU).

Each test checks the oracle against something other than itself: hand-worked
groups, the half-step error bound stated by the axis-selection guide
("量化错误的真正组成"), exact brute force over all levels, and the isolation
property that motivates the grouping axes (keys: fixed outlier channels;
values: per-token groups).
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant


def _parse(line):
    B, xs, s, z, codes, xhat = [p.strip() for p in line.split(";")]
    f16 = lambda t: np.array([float(v) for v in t.split()], np.float16)
    return (int(B), f16(xs), np.float16(float(s)), np.float16(float(z)),
            np.array([int(c) for c in codes.split()]), np.array([float(v) for v in xhat.split()]))


def test_worked_examples(golden):
    lines = golden("quantizer_worked_examples.txt")
    assert len(lines) == 6
    for line in lines:
        B, x, s, z, codes, xhat = _parse(line)
        c, s_o, z_o = quant.quantize_groups(x, B, axis=0)
        assert c.tolist() == codes.tolist(), line
        assert s_o[0].tobytes() == s.tobytes(), line          # bit-exact, +0 included
        assert z_o[0].tobytes() == z.tobytes(), line
        np.testing.assert_array_equal(quant.dequantize(c, s_o, z_o), xhat)


def test_zero_point_sign_is_canonical():
    x = np.array([-0.0, -0.0, 1.0, 2.0], np.float16)
    _, _, z = quant.quantize_groups(x, 2, axis=0)
    assert z.view(np.uint16)[0] == 0                         # +0, not -0


def _exact_nearest(x, s, z, L):
    """Exact distances to every level k*s + z, k = 0..L (fractions)."""
    xs, ss, zs = Fraction(float(x)), Fraction(float(s)), Fraction(float(z))
    return [abs(xs - (k * ss + zs)) for k in range(L + 1)]


@pytest.mark.parametrize("B", [2, 4, 8])
def test_brute_force_nearest_level(B):
    """Each chosen code is a nearest level of the stored grid (exact arithmetic).

    fp32 rounding of (x - z) and of its quotient by s moves the ratio by at
    most 2^-23 of its size (< L + 1), so the farther neighbour can be picked
    only that close to a half-integer: the allowed excess distance is
    s * max(2^-18, (L + 1) * 2^-22).
    """
    rng = np.random.default_rng(7)
    L = quant.levels(B)
    for G in (2, 3, 5, 8):
        X = (rng.standard_normal((400, G)) * rng.uniform(0.01, 30, (400, 1))).astype(np.float16)
        codes, s, z = quant.quantize_groups(X, B, axis=1)
        for g in range(X.shape[0]):
            for j in range(G):
                d = _exact_nearest(X[g, j], s[g, 0], z[g, 0], L)
                assert 0 <= codes[g, j] <= L
                slack = Fraction(float(s[g, 0])) * max(Fraction(1, 2**18), Fraction(L + 1, 2**22))
                assert d[codes[g, j]] <= min(d) + slack


@pytest.mark.parametrize("B", [2, 4])
def test_joint_brute_force_small_groups(B):
    """Over all (L+1)^G code vectors, the chosen one minimizes the squared error."""
    import itertools
    rng = np.random.default_rng(11)
    L = quant.levels(B)
    G = 3 if B == 4 else 4
    X = (rng.standard_normal((30, G)) * 3).astype(np.float16)
    codes, s, z = quant.quantize_groups(X, B, axis=1)
    for g in range(X.shape[0]):
        ss, zs = Fraction(float(s[g, 0])), Fraction(float(z[g, 0]))
        xs = [Fraction(float(v)) for v in X[g]]
        err = lambda cv: sum((x - (c * ss + zs)) ** 2 for x, c in zip(xs, cv))
        best = min(err(cv) for cv in itertools.product(range(L + 1), repeat=G))
        assert err(codes[g]) <= best + G * (ss / 2**17) ** 2 + 2 * G * ss * ss / 2**18


@pytest.mark.parametrize("B", [2, 4, 8])
def test_half_step_bound_and_level_coverage(B):
    """|x - x_hat| <= s/2 (+ fp32 slack); the minimum gets code 0 and the maximum code L."""
    rng = np.random.default_rng(3)
    L = quant.levels(B)
    X = (rng.standard_normal((2000, 32)) * rng.uniform(0.5, 50, (2000, 1))).astype(np.float16)
    codes, s, z = quant.quantize_groups(X, B, axis=1)
    xhat = quant.dequantize(codes, s, z)
    sd = s.astype(np.float64)
    err = np.abs(X.astype(np.float64) - xhat)
    assert np.all(err <= sd / 2 * (1 + max(2.0**-17, (L + 1) * 2.0**-21)))
    assert np.all(s > 0)
    assert np.all(codes[np.arange(2000), X.argmin(axis=1)] == 0)
    assert np.all(codes[np.arange(2000), X.argmax(axis=1)] == L)
    # the stored step is the fp16 rounding of range / L
    rng_ = X.max(axis=1).astype(np.float64) - X.min(axis=1).astype(np.float64)
    assert np.all(np.abs(sd[:, 0] - rng_ / L) <= rng_ / L * 2.0**-11 * 1.0001)


def test_key_grouping_isolates_outlier_channel():
    """Per-channel key groups: an x1000 channel does not inflate other channels' steps.

    Grouping keys along the token axis per channel ([axis-guide] keys section)
    bounds each ordinary channel's error by half of ITS OWN step.
    """
    rng = np.random.default_rng(5)
    l, d, G = 64, 32, 16
    K = rng.standard_normal((l, d)).astype(np.float32)
    K[:, 7] *= 1000
    K = K.astype(np.float16)
    codes, s, z = quant.quantize_keys(K, 2, G)
    assert codes.shape == (l, d) and s.shape == (l // G, d) and z.shape == (l // G, d)
    err = np.abs(K.astype(np.float64) - quant.dequantize_keys(codes, s, z, G))
    for g in range(l // G):
        blk = K[g * G:(g + 1) * G].astype(np.float64)
        own = (blk.max(axis=0) - blk.min(axis=0)) / 3
        assert np.all(err[g * G:(g + 1) * G] <= own / 2 * (1 + 2.0**-9) + 1e-12)
    # ordinary channels' errors stay far below the outlier channel's step
    ordinary = np.delete(err, 7, axis=1)
    assert ordinary.max() < 0.01 * s[:, 7].astype(np.float64).min()


def test_value_grouping_isolates_outlier_token():
    """Per-token value groups: an x1000 token does not touch other tokens' errors."""
    rng = np.random.default_rng(6)
    l, d, G = 20, 64, 32
    V = rng.standard_normal((l, d)).astype(np.float32)
    V[4] *= 1000
    V = V.astype(np.float16)
    codes, s, z = quant.quantize_values(V, 2, G)
    assert s.shape == (l, d // G)
    err = np.abs(V.astype(np.float64) - quant.dequantize_values(codes, s, z, G))
    for t in range(l):
        for j in range(d // G):
            seg = V[t, j * G:(j + 1) * G].astype(np.float64)
            own = (seg.max() - seg.min()) / 3
            assert np.all(err[t, j * G:(j + 1) * G] <= own / 2 * (1 + 2.0**-9))
    assert np.delete(err, 4, axis=0).max() < 2.0


def test_outlier_channels_favour_per_channel_keys():
    """Direction of the key result in [axis-guide] (keys section): with fixed
    outlier channels, per-channel grouping gives a smaller attention-score
    error than per-token grouping of the same keys."""
    rng = np.random.default_rng(9)
    l, d, G = 256, 128, 32
    K = rng.standard_normal((l, d)).astype(np.float32)
    # outlier channels: a very large magnitude on every token, same channels throughout
    K[:, [3, 50, 77, 100]] += np.array([40.0, -55.0, 30.0, 70.0], np.float32)
    K = K.astype(np.float16)
    q = rng.standard_normal(d)
    kc, ks, kz = quant.quantize_keys(K, 2, G)
    per_channel = quant.dequantize_keys(kc, ks, kz, G)
    # per-token grouping of keys: transpose the roles
    tc, ts, tz = quant.quantize_values(K, 2, G)
    per_token = quant.dequantize_values(tc, ts, tz, G)
    exact = K.astype(np.float64) @ q
    e_ch = np.abs(per_channel @ q - exact).mean()
    e_tok = np.abs(per_token @ q - exact).mean()
    assert e_ch < e_tok / 2
