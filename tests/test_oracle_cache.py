"""Pins for the oracle's streaming cache: prefill split, residual, flush (no GPU)."""
import numpy as np
import pytest

from oracle import quant
from oracle.cache import OracleCache, prefill_split


def _tokens(rng, B, H, n, d):
    K = rng.standard_normal((B, H, n, d)).astype(np.float32)
    K[..., 5] *= 25
    return K.astype(np.float16), rng.standard_normal((B, H, n, d)).astype(np.float16)


def test_prefill_split_rule():
    # the quantized prefix is whole groups and leaves at most R tokens in fp16
    assert prefill_split(256, 32, 32) == (224, 32)     # tiny workload: 224 of 256 quantized
    assert prefill_split(4096, 32, 128) == (3968, 128)
    assert prefill_split(8192, 128, 128) == (8064, 128)
    assert prefill_split(131072, 32, 128) == (130944, 128)
    assert prefill_split(0, 32, 128) == (0, 0)
    assert prefill_split(100, 32, 128) == (0, 100)
    assert prefill_split(129, 32, 128) == (32, 97)
    for l in range(0, 600):
        for G, R in ((32, 32), (32, 128), (64, 128), (128, 128)):
            Lq, r = prefill_split(l, G, R)
            assert Lq % G == 0 and 0 <= r <= R and Lq + r == l
            # the smallest such prefix: one group less would leave more than R
            assert Lq == 0 or l - (Lq - G) > R


@pytest.mark.parametrize("G,R,L0,n", [(32, 32, 256, 1), (32, 128, 300, 300), (16, 64, 0, 150),
                                      (64, 128, 129, 260), (32, 64, 64, 1)])
def test_streaming_equals_one_shot(G, R, L0, n):
    """After prefill(L0) and n appends the quantized part equals a one-shot
    quantization of the same token prefix (group boundaries at multiples of G
    from token 0) and the residual holds the remaining tokens bit for bit."""
    rng = np.random.default_rng(G + R + L0 + n)
    B, H, d, bits = 2, 3, 64, 2
    K, V = _tokens(rng, B, H, L0 + n, d)
    c = OracleCache(B, H, d, bits, G, R)
    c.prefill(K[:, :, :L0], V[:, :, :L0])
    flushes_expected = 0
    r = c.n_resid
    for t in range(L0, L0 + n):
        if r == R:
            flushes_expected += 1
            r = 0
        c.append(K[:, :, t], V[:, :, t])
        r += 1
        assert c.n_quant + c.n_resid == t + 1
        assert c.n_quant % G == 0 and 1 <= c.n_resid <= R
    assert c.flushes == flushes_expected
    Lq = c.n_quant
    kc, ks, kz = quant.quantize_keys(K[:, :, :Lq], bits, G)
    vc, vs, vz = quant.quantize_values(V[:, :, :Lq], bits, G)
    for a, b in ((c.k_codes, kc), (c.k_s, ks), (c.k_z, kz), (c.v_codes, vc), (c.v_s, vs), (c.v_z, vz)):
        assert a.tobytes() == b.tobytes()
    assert c.k_res.tobytes() == np.ascontiguousarray(K[:, :, Lq:]).tobytes()
    assert c.v_res.tobytes() == np.ascontiguousarray(V[:, :, Lq:]).tobytes()


def test_flush_is_lazy_and_counts():
    rng = np.random.default_rng(1)
    K, V = _tokens(rng, 1, 1, 256 + 70, 64)
    c = OracleCache(1, 1, 64, 2, 32, 32)
    c.prefill(K[:, :, :256], V[:, :, :256])
    assert (c.n_quant, c.n_resid) == (224, 32)          # full residual at rest
    c.append(K[:, :, 256], V[:, :, 256])
    assert (c.n_quant, c.n_resid, c.flushes) == (256, 1, 1)
    for t in range(257, 256 + 70):
        c.append(K[:, :, t], V[:, :, t])
    # flushes happen when the residual is found full: n appends after a full
    # residual of R give ceil(n / R) flushes
    assert c.flushes == -(-70 // 32)
    assert c.n_quant + c.n_resid == 326


def test_prefill_twice_rejected():
    c = OracleCache(1, 1, 32, 2, 32, 32)
    K = np.zeros((1, 1, 40, 32), np.float16)
    c.prefill(K, K)
    with pytest.raises(RuntimeError):
        c.prefill(K, K)


def test_dequantized_cache_matches_inputs_within_half_step():
    rng = np.random.default_rng(2)
    K, V = _tokens(rng, 1, 2, 200, 64)
    c = OracleCache(1, 2, 64, 4, 32, 64)
    c.prefill(K, V)
    kh, vh = c.keys_hat(), c.values_hat()
    Lq = c.n_quant
    ks = np.repeat(c.k_s, 32, axis=2).astype(np.float64)
    vs = np.repeat(c.v_s, 32, axis=3).astype(np.float64)
    assert np.all(np.abs(kh[:, :, :Lq] - K[:, :, :Lq]) <= ks / 2 * (1 + 2.0**-17))
    assert np.all(np.abs(vh[:, :, :Lq] - V[:, :, :Lq]) <= vs / 2 * (1 + 2.0**-17))
    # residual rows are the exact fp16 inputs
    assert np.array_equal(kh[:, :, Lq:], K[:, :, Lq:].astype(np.float64))


# ---- the value queue of [explainer] 3.2 (OracleCacheFifo) ---------------------------------

from oracle.cache import OracleCacheFifo  # noqa: E402


def _stream(cache, K, V, L0):
    cache.prefill(K[:, :, :L0], V[:, :, :L0])
    for t in range(L0, K.shape[2]):
        cache.append(K[:, :, t], V[:, :, t])


@pytest.mark.parametrize("G,R,L0,n", [(32, 32, 256, 5), (32, 128, 300, 300), (16, 64, 0, 150),
                                      (64, 128, 129, 260), (32, 64, 40, 30)])
def test_fifo_values_equal_one_shot_per_token(G, R, L0, n):
    """The quantized values are a one-shot per-token quantization of the first
    max(l - R, 0) tokens; the queue holds the newest min(l, R) values bit for
    bit; the keys are those of the flush-all cache."""
    rng = np.random.default_rng(7 + G + R + L0 + n)
    B, H, d, bits = 1, 2, 64, 2
    K, V = _tokens(rng, B, H, L0 + n, d)
    fifo, flush = OracleCacheFifo(B, H, d, bits, G, R), OracleCache(B, H, d, bits, G, R)
    _stream(fifo, K, V, L0)
    _stream(flush, K, V, L0)
    l = L0 + n
    Lv = max(l - R, 0)
    assert fifo.n_quant_v == Lv and fifo.v_res.shape[2] == min(l, R)
    vc, vs, vz = quant.quantize_values(V[:, :, :Lv], bits, G)
    assert np.array_equal(fifo.v_codes, vc) and np.array_equal(fifo.v_s.view(np.uint16), vs.view(np.uint16))
    assert np.array_equal(fifo.v_z.view(np.uint16), vz.view(np.uint16))
    assert fifo.v_res.tobytes() == V[:, :, Lv:].tobytes()
    assert np.array_equal(fifo.keys_hat(), flush.keys_hat())
    assert (fifo.n_quant, fifo.n_resid) == (flush.n_quant, flush.n_resid)
    vh = fifo.values_hat()
    assert vh.shape[2] == l
    assert np.array_equal(vh[:, :, Lv:], V[:, :, Lv:].astype(np.float64))


def test_fifo_hand_worked_positions():
    """d = 4, G = 2, R = 2: after a 3-token prompt token 0 is quantized and
    tokens 1, 2 wait; each append pops one more; the keys flush two at a time."""
    G, R, d = 2, 2, 4
    c = OracleCacheFifo(1, 1, d, 2, G, R)
    K = np.arange(6 * d, dtype=np.float16).reshape(1, 1, 6, d)
    V = (np.arange(6 * d, dtype=np.float16) * 0.5).reshape(1, 1, 6, d)
    c.prefill(K[:, :, :3], V[:, :, :3])
    assert (c.n_quant, c.n_resid, c.n_quant_v, c.v_res.shape[2]) == (2, 1, 1, 2)
    assert c.v_res.tobytes() == V[:, :, 1:3].tobytes()
    c.append(K[:, :, 3], V[:, :, 3])           # key residual 1 -> 2; value 1 popped
    assert (c.n_quant, c.n_resid, c.n_quant_v) == (2, 2, 2)
    c.append(K[:, :, 4], V[:, :, 4])           # key flush of tokens 2, 3; value 2 popped
    assert (c.n_quant, c.n_resid, c.n_quant_v) == (4, 1, 3)
    assert c.v_res.tobytes() == V[:, :, 3:5].tobytes()
    # token 0's values 0, .5, 1, 1.5 in groups (0, .5), (1, 1.5): step .5 / 3 per group
    assert c.v_codes[0, 0, 0].tolist() == [0, 3, 0, 3]
    assert c.v_z[0, 0, 0].tolist() == [0.0, 1.0]


def test_fifo_values_exact_in_the_window_where_flush_quantizes():
    """Right after a flush of the flush-all cache, its R newest tokens but one
    are quantized, while the queue still has them in fp16: the two caches'
    values differ exactly on [l - R, l - 1) and agree elsewhere."""
    rng = np.random.default_rng(3)
    B, H, d, bits, G, R = 1, 1, 64, 2, 32, 64
    K, V = _tokens(rng, B, H, 64 + 65, d)
    fifo, flush = OracleCacheFifo(B, H, d, bits, G, R), OracleCache(B, H, d, bits, G, R)
    _stream(fifo, K, V, 64)
    _stream(flush, K, V, 64)                   # the 65th append flushed 64 tokens
    l = K.shape[2]
    vf, vq = fifo.values_hat(), flush.values_hat()
    diff = np.any(vf != vq, axis=-1)[0, 0]
    assert not diff[: l - R].any() and not diff[l - 1]
    assert diff[l - R: l - 1].all()
