"""The benchmark's algorithmic byte and token counts (the roofline's numerator
and the metric's token count) against the oracle's closed-form accounting,
which is pinned to the explainer's fp16 figure and hand-worked per-token bytes
(no GPU)."""
import pytest

import bench
from oracle import accounting
from oracle.cache import prefill_split


def _last_state(L, n, G, R):
    """(Lq, r) of a sequence after a prompt of L tokens and n appends (flush-all rule)."""
    Lq, r = prefill_split(L, G, R)
    for _ in range(n):
        if r == R:
            Lq, r = Lq + R, 0
        r += 1
    return Lq, r


@pytest.mark.parametrize("name", ["tiny-b1h1d64", "llama2-7b-layer", "llama2-13b-40layer", "llama3-8b-gqa",
                                  "long-context", "llama2-7b-layer-8bit"])
def test_dense_call_bytes_match_the_oracle(name):
    w = bench.WORKLOADS[name]
    Lq, r = _last_state(w["prompt"], w["decode"], w["G"], w["R"])
    want = accounting.decode_call_bytes(w["B"], w["Hq"], w["Hkv"], w["D"], w["bits"], w["G"], Lq, r)
    assert bench._bytes_last_call(w) == want
    assert bench._tokens_last_call(w) == w["B"] * (Lq + r)


def test_seven_b_closed_forms():
    w = bench.WORKLOADS["llama2-7b-layer"]
    # prompt 4096 -> 3968 quantized + 128 residual; the first append flushes; 64 appends -> (4096, 64)
    assert _last_state(4096, 64, 32, 128) == (4096, 64)
    assert bench._bytes_last_call(w) == 256 * (4096 * 96 + 64 * 512) + 2 * 8 * 32 * 128 * 2 == 109_182_976
    # tokens attended per step: 4 layers x 8 rows x sum over the 64 calls of (4096 + s)
    assert bench._kv_tokens_per_step(w) == 4 * 8 * sum(4096 + s for s in range(1, 65))


def test_ragged_call_bytes_are_the_sum_over_sequences():
    w = bench.WORKLOADS["llama2-7b-ragged"]
    total, toks = 0, 0
    for L in w["lengths"]:
        Lq, r = _last_state(L, w["decode"], w["G"], w["R"])
        total += accounting.decode_call_bytes(1, w["Hq"], w["Hkv"], w["D"], w["bits"], w["G"], Lq, r)
        toks += Lq + r
    assert bench._bytes_last_call(w) == total
    assert bench._tokens_last_call(w) == toks


def test_value_queue_call_bytes():
    """Keys quantized over Lq tokens, values over the first L - R; the rest fp16."""
    w = bench.WORKLOADS["llama2-7b-layer-vqueue"]
    Lq, r = _last_state(w["prompt"], w["decode"], w["G"], w["R"])
    L = Lq + r
    Lv = max(L - w["R"], 0)
    half = accounting.quantized_bytes_per_token(w["D"], w["bits"], w["G"]) // 2   # K or V part per token
    per_slot = Lq * half + Lv * half + r * 2 * w["D"] + (L - Lv) * 2 * w["D"]
    want = w["B"] * w["Hkv"] * per_slot + 2 * w["B"] * w["Hq"] * w["D"] * 2
    assert bench._bytes_last_call(w) == want
