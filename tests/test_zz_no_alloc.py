"""Decode with the library-owned static workspace (kivi_decode_attn_static_ws).

That entry point serves callers that cannot allocate device memory (a plugin
whose host framework owns all device memory, code that is only handed device
pointers).  It runs the same kernels on the same grid as kivi_decode_attn with
a caller workspace, so its output must be the same bit for bit, call after
call, although every call reuses one workspace that keeps the last call's
partial results.  After the first call on a device (which loads the array),
no call may change the device's free memory.  This file is named so that
pytest collects it last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU hosts too
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_kivi_kv_gb300 import kivi as K  # noqa: E402
from bit_kivi_kv_gb300.synth import SynthKV  # noqa: E402


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _static(cache, q, out):
    K.kivi_decode_attn_static_ws(cache.handle, q.data_ptr(), out.data_ptr(), 0.0, _stream())


def _cache(B, Hq, Hkv, D, bits, G, R, L, seed, extra=8):
    syn = SynthKV(B, Hq, Hkv, D, seed=seed, device="cuda")
    Kp, Vp = syn.prompt(L)
    cache = K.KiviCache(B, Hq, Hkv, D, bits, G, R, L + extra)
    cache.prefill(Kp, Vp)
    return cache, syn


def test_static_workspace_matches_caller_workspace_on_consecutive_calls():
    cache, syn = _cache(4, 8, 4, 128, 2, 32, 128, 1000, seed=77)
    for s in range(2):                                  # two calls in a row, different contexts
        q, k, v = syn.step(s)
        cache.append(k, v)
        ref = cache.decode_attn(q)
        got = torch.full_like(q, float("nan"))
        _static(cache, q, got)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)
    # two back-to-back calls with different queries on the same cache state
    q1, q2 = syn.step(10)[0], syn.step(11)[0]
    g1, g2 = torch.empty_like(q1), torch.empty_like(q2)
    _static(cache, q1, g1)
    _static(cache, q2, g2)
    r1, r2 = cache.decode_attn(q1), cache.decode_attn(q2)
    torch.cuda.synchronize()
    assert torch.equal(g1, r1)
    assert torch.equal(g2, r2)


def test_static_workspace_long_then_short_context_on_another_cache():
    # the long context leaves more partial results per head in the shared
    # workspace than the short one reads back; stale ones must not leak in
    long_c, long_syn = _cache(2, 8, 8, 128, 2, 32, 128, 20000, seed=91)
    short_c, short_syn = _cache(2, 8, 8, 128, 2, 32, 128, 300, seed=92)
    ql, qs = long_syn.step(0)[0], short_syn.step(0)[0]
    gl, gs = torch.empty_like(ql), torch.empty_like(qs)
    _static(long_c, ql, gl)
    _static(short_c, qs, gs)
    rl, rs = long_c.decode_attn(ql), short_c.decode_attn(qs)
    torch.cuda.synchronize()
    assert torch.equal(gl, rl)
    assert torch.equal(gs, rs)


def test_static_workspace_calls_allocate_nothing():
    cache, syn = _cache(2, 8, 8, 128, 4, 64, 128, 2000, seed=93)
    qs = [syn.step(s)[0] for s in range(3)]
    outs = [torch.empty_like(q) for q in qs]
    _static(cache, qs[0], outs[0])                      # the first call on the device loads the array
    torch.cuda.synchronize()
    reserved = torch.cuda.memory_reserved()
    free0, _ = torch.cuda.mem_get_info()
    for q, o in zip(qs, outs):
        _static(cache, q, o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_reserved() == reserved
    assert free1 == free0
    for q, o in zip(qs, outs):
        assert torch.equal(o, cache.decode_attn(q))


def test_static_workspace_rejects_shapes_beyond_its_size():
    # 64 x 32 query heads at head_dim 128 need about 70 MB of workspace (> 16 MiB)
    cache, syn = _cache(64, 32, 8, 128, 4, 128, 128, 200, seed=5)
    q = syn.step(0)[0]
    out = torch.empty_like(q)
    with pytest.raises(K.KiviError) as e:
        _static(cache, q, out)
    assert e.value.status == K.KIVI_ERR_CAPACITY
    assert "static" in str(e.value)
