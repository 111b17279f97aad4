"""Many live handles in one process.

A model keeps one cache handle per layer, so a process holds tens of handles of
possibly different shapes, each with its own host state, while the kernels'
per-instance launch set-up is shared by every handle of a shape.  Here nine
handles of different head dims, bit widths, groups, query-head ratios, decode
kernels and value-residual modes are created together and then driven
interleaved: every step calls every handle, in an order that rotates, some with
the fused append + decode and some with the two separate calls.  Each handle's
outputs at three steps and its cache bytes at the end must match its own oracle
replay, and every buffer's guard bands must be intact.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU hosts too
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_kivi_kv_gb300.kivi import KIVI_DECODE_CUDA_CORE, KIVI_DECODE_TENSOR_CORE  # noqa: E402
from bit_kivi_kv_gb300.synth import SynthKV  # noqa: E402
from guards import GuardedCache  # noqa: E402
from kivi_harness import check_slots, run_gpu  # noqa: E402

TC, CC = KIVI_DECODE_TENSOR_CORE, KIVI_DECODE_CUDA_CORE
HANDLES = [
    # B, Hq, Hkv, D, bits, G, R, prompt, decode kernel, value queue
    (2, 8, 8, 128, 2, 32, 128, 900, TC, False),
    (2, 8, 2, 128, 4, 128, 128, 1300, TC, False),
    (1, 4, 4, 64, 2, 32, 64, 300, TC, False),
    (2, 4, 2, 64, 8, 64, 64, 500, TC, False),
    (1, 8, 8, 128, 8, 32, 32, 700, TC, False),
    (2, 8, 8, 128, 2, 32, 128, 900, CC, False),   # the CUDA-core kernel on the first handle's shape
    (1, 8, 4, 128, 2, 64, 128, 1000, TC, True),
    (3, 6, 3, 64, 4, 32, 32, 250, TC, False),
    (1, 16, 4, 128, 4, 32, 64, 2000, TC, False),
]


def test_many_live_handles_interleaved():
    n = 40
    decode_at = {0, 17, 39}
    runs = []
    for i, (B, Hq, Hkv, D, bits, G, R, L, kernel, vqueue) in enumerate(HANDLES):
        syn = SynthKV(B, Hq, Hkv, D, 3000 + i, device="cuda")
        K, V = syn.prompt(L)
        cache = GuardedCache(B, Hq, Hkv, D, bits, G, R, L + n)
        cache.set_decode_kernel(kernel)
        if vqueue:
            cache.set_value_residual(1)
        cache.prefill(K, V)
        runs.append(dict(cache=cache, syn=syn, K=K, V=V, steps=[], outs={}, B=B, Hq=Hq, Hkv=Hkv, D=D,
                         bits=bits, G=G, R=R, L=L, vqueue=vqueue))
    for s in range(n):
        order = runs[s % len(runs):] + runs[:s % len(runs)]
        for j, run in enumerate(order):
            q, k, v = run["syn"].step(s)
            run["steps"].append((q, k, v))
            cache = run["cache"]
            if s not in decode_at:
                cache.append(k, v)
                continue
            out = cache.bands.like(q)
            if (j + s) % 2:
                run["outs"][s] = cache.append_decode(k, v, q, out=out)
            else:
                cache.append(k, v)
                run["outs"][s] = cache.decode_attn(q, out=out)
    torch.cuda.synchronize()
    for i, run in enumerate(runs):
        run["cache"].bands.check(f"handle {i} after the interleaved calls")
        run["outs"] = {s: o.cpu() for s, o in run["outs"].items()}
        check_slots(run, [(0, 0), (run["B"] - 1, run["Hkv"] - 1)], decode_at)


def test_llama2_13b_forty_layers_full_size():
    """The 13B configuration as a step: 40 live layer caches (B32 H40 D128, 2-bit,
    G32, R128; ~0.5 GB each), each prefilled with its own 4096-token prompt, then
    one fused append + decode through all 40 layers with a fresh query per layer
    (each append flushes its layer's full residual).  Four layers, spread over
    the stack, are checked slot by slot against the oracle; the others must give
    finite outputs and the expected token counts."""
    from bit_kivi_kv_gb300.kivi import KiviCache
    B, H, D, L, n_layers = 32, 40, 128, 4096, 40
    checked = {0, 13, 26, 39}
    runs, outs = {}, []
    caches = []
    for li in range(n_layers):
        if li in checked:
            # a checked layer keeps its prompt and step for the oracle
            runs[li] = run_gpu(B, H, H, D, 2, 32, 128, L, 0, seed=5000 + li, max_tokens=L + 1)
            caches.append(runs[li]["cache"])
            continue
        syn = SynthKV(B, H, H, D, 5000 + li, device="cuda")
        K, V = syn.prompt(L)
        c = KiviCache(B, H, H, D, 2, 32, 128, L + 1)
        c.prefill(K, V)
        del K, V
        caches.append(c)
    for li, c in enumerate(caches):
        if li in checked:
            syn = SynthKV(B, H, H, D, 5000 + li, device="cuda")
            q, k, v = syn.step(0)
            runs[li]["steps"].append((q, k, v))
            runs[li]["outs"][0] = c.append_decode(k, v, q)
        else:
            q, k, v = SynthKV(B, H, H, D, 9000 + li, device="cuda").step(0)
            outs.append(c.append_decode(k, v, q))
    torch.cuda.synchronize()
    for c in caches:
        assert c.counts() == (L, 1)
    for o in outs:
        assert torch.isfinite(o.float()).all()
    for li, run in runs.items():
        run["outs"] = {s: o.cpu() for s, o in run["outs"].items()}
        check_slots(run, [(0, 0), (17, 23), (31, 39)], {0})
