"""Pins for the oracle's fp64 decode attention (no GPU): closed forms and invariants."""
import math

import numpy as np

from oracle.attention import decode_attention


def _rand(seed, B=2, Hq=2, Hkv=2, T=37, d=16):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, d)), rng.standard_normal((B, Hkv, T, d)) * 2,
            rng.standard_normal((B, Hkv, T, d)))


def test_zero_query_gives_mean():
    _, K, V = _rand(0)
    q = np.zeros((2, 2, 16))
    o, lse = decode_attention(q, K, V)
    np.testing.assert_allclose(o, V.mean(axis=2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(37), rtol=0, atol=1e-13)


def test_two_tokens_logistic_closed_form():
    rng = np.random.default_rng(1)
    d = 8
    q = rng.standard_normal((1, 1, d))
    K = rng.standard_normal((1, 1, 2, d))
    V = rng.standard_normal((1, 1, 2, d))
    o, _ = decode_attention(q, K, V, scale=0.7)
    delta = 0.7 * float(q[0, 0] @ (K[0, 0, 1] - K[0, 0, 0]))
    w1 = 1.0 / (1.0 + math.exp(-delta))
    np.testing.assert_allclose(o[0, 0], w1 * V[0, 0, 1] + (1 - w1) * V[0, 0, 0], atol=1e-14)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(2)
    V = rng.standard_normal((1, 1, 1, 8))
    o, _ = decode_attention(rng.standard_normal((1, 1, 8)), rng.standard_normal((1, 1, 1, 8)), V)
    np.testing.assert_array_equal(o[0, 0], V[0, 0, 0])


def test_dominant_token_bound():
    """One logit above all others by D: |o - v0| <= (T-1) e^{-D} * 2 max|v|."""
    rng = np.random.default_rng(3)
    T, d = 50, 16
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    K = rng.uniform(-1, 1, (1, 1, T, d)); K[0, 0, :, 0] = 0.0
    K[0, 0, 0, 0] = 12.0
    V = rng.standard_normal((1, 1, T, d))
    o, _ = decode_attention(q, K, V, scale=1.0)
    gap = 12.0
    bound = (T - 1) * math.exp(-gap) * 2 * np.abs(V).max()
    assert np.abs(o[0, 0] - V[0, 0, 0]).max() <= bound


def test_permutation_invariance():
    q, K, V = _rand(4)
    perm = np.random.default_rng(5).permutation(K.shape[2])
    o1, l1 = decode_attention(q, K, V)
    o2, l2 = decode_attention(q, K[:, :, perm], V[:, :, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_logit_shift_invariance():
    """Adding c*q/|q|^2 to every key shifts every logit by scale*c: o unchanged."""
    q, K, V = _rand(6, B=1, Hq=1, Hkv=1)
    qq = q[0, 0]
    K2 = K + 5.0 * qq / (qq @ qq)
    o1, l1 = decode_attention(q, K, V, scale=0.5)
    o2, l2 = decode_attention(q, K2, V, scale=0.5)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 2.5, atol=1e-12)


def test_grouped_query_equals_replicated_heads():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 8, 16))
    K = rng.standard_normal((2, 2, 21, 16))
    V = rng.standard_normal((2, 2, 21, 16))
    o_g, _ = decode_attention(q, K, V)
    o_m, _ = decode_attention(q, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1))
    np.testing.assert_array_equal(o_g, o_m)


def test_default_scale_and_explicit_scale():
    q, K, V = _rand(8)
    o1, _ = decode_attention(q, K, V)                      # 1/sqrt(16) = 0.25
    o2, _ = decode_attention(q * 0.5, K, V, scale=0.5)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
