"""Decode with the library-owned static workspace (kivi_decode_attn_static_ws).

That entry point serves callers that cannot allocate device memory (a plugin
whose host framework owns all device memory, code that is only handed device
pointers).  It must give the same output as kivi_decode_attn with a caller
workspace, call after call, although every call reuses one workspace.  This
file is named so that pytest collects it last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU hosts too
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_kivi_kv_gb300 import kivi as K  # noqa: E402
from bit_kivi_kv_gb300.synth import SynthKV  # noqa: E402
from kivi_harness import ATOL, RTOL_L2  # noqa: E402


def _close(a, b):
    a, b = a.double(), b.double()
    err = (a - b).abs()
    assert err.max().item() <= ATOL
    assert (err.norm() / b.norm()).item() <= RTOL_L2


def test_static_workspace_matches_caller_workspace_on_consecutive_calls():
    B, Hq, Hkv, D, bits, G, R, L = 4, 8, 4, 128, 2, 32, 128, 1000
    syn = SynthKV(B, Hq, Hkv, D, seed=77, device="cuda")
    Kp, Vp = syn.prompt(L)
    cache = K.KiviCache(B, Hq, Hkv, D, bits, G, R, L + 8)
    cache.prefill(Kp, Vp)
    stream = torch.cuda.current_stream().cuda_stream
    for s in range(2):                                  # two calls in a row, different contexts
        q, k, v = syn.step(s)
        cache.append(k, v)
        ref = cache.decode_attn(q)
        got = torch.full_like(q, float("nan"))
        K.kivi_decode_attn_static_ws(cache.handle, q.data_ptr(), got.data_ptr(), 0.0, stream)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        _close(got, ref)
    # two back-to-back calls with different queries on the same cache state
    q1, q2 = syn.step(10)[0], syn.step(11)[0]
    g1, g2 = torch.empty_like(q1), torch.empty_like(q2)
    K.kivi_decode_attn_static_ws(cache.handle, q1.data_ptr(), g1.data_ptr(), 0.0, stream)
    K.kivi_decode_attn_static_ws(cache.handle, q2.data_ptr(), g2.data_ptr(), 0.0, stream)
    r1, r2 = cache.decode_attn(q1), cache.decode_attn(q2)
    torch.cuda.synchronize()
    _close(g1, r1)
    _close(g2, r2)


def test_static_workspace_rejects_shapes_beyond_its_size():
    # 64 x 32 query heads at head_dim 128 need about 70 MB of workspace (> 16 MiB)
    cache = K.KiviCache(64, 32, 8, 128, 4, 128, 128, 256)
    syn = SynthKV(64, 32, 8, 128, seed=5, device="cuda")
    Kp, Vp = syn.prompt(200)
    cache.prefill(Kp, Vp)
    q = syn.step(0)[0]
    out = torch.empty_like(q)
    with pytest.raises(K.KiviError) as e:
        K.kivi_decode_attn_static_ws(cache.handle, q.data_ptr(), out.data_ptr(), 0.0,
                                     torch.cuda.current_stream().cuda_stream)
    assert e.value.status == K.KIVI_ERR_CAPACITY
    assert "static" in str(e.value)
