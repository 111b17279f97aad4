"""Shared helpers for the GPU parity tests: run a workload through the C ABI,
rebuild the same slots with the CPU oracle, compare bytes and outputs."""
from __future__ import annotations

import numpy as np
import torch

from bit_kivi_kv_gb300.kivi import kivi_cache_set_max_ctas
from bit_kivi_kv_gb300.synth import RANGE_2_6_X10_50, SynthKV
from guards import GuardedCache
from oracle import layout
from oracle.attention import decode_attention
from oracle.cache import OracleCache, OracleCacheFifo

ATOL = 4e-3      # max |out - oracle|
RTOL_L2 = 1e-3   # ||out - oracle||_2 / ||oracle||_2


def run_gpu(B, Hq, Hkv, D, bits, G, R, L, n_app, seed, decode_at=(), outliers=RANGE_2_6_X10_50,
            sink=True, max_tokens=None, prompt=None, decode_kernel=0, fused=False, vqueue=False,
            max_ctas=0):
    """Prefill L tokens, then n_app x append (decoding at the steps in decode_at;
    with fused, those steps append and decode in one kivi_append_decode call,
    fused may also be the set of steps that do; with vqueue, the cache keeps
    its value residual as a queue; max_ctas caps the decode grid).

    The cache buffer, the workspace and every output sit between guard bands,
    checked after every call.
    Returns dict(cache, K, V, steps=[(q,k,v)], outs={step: out fp16 cpu}).
    """
    syn = SynthKV(B, Hq, Hkv, D, seed, outliers=outliers, sink=sink, device="cuda")
    K, V = prompt if prompt is not None else syn.prompt(L)
    cache = GuardedCache(B, Hq, Hkv, D, bits, G, R, max_tokens or max(L + n_app, 1))
    cache.set_decode_kernel(decode_kernel)
    if max_ctas:
        kivi_cache_set_max_ctas(cache.handle, max_ctas)
    if vqueue:
        cache.set_value_residual(1)
    cache.prefill(K, V)
    cache.bands.check("after the prefill")
    steps, outs = [], {}
    for s in range(n_app):
        q, k, v = syn.step(s)
        steps.append((q, k, v))
        fuse = (s in fused) if isinstance(fused, (set, frozenset)) else fused
        if fuse and s in decode_at:
            out = cache.bands.like(q)
            outs[s] = cache.append_decode(k, v, q, out=out).cpu()
            cache.bands.check(f"after the fused call of step {s}")
            continue
        cache.append(k, v)
        if s in decode_at:
            out = cache.bands.like(q)
            outs[s] = cache.decode_attn(q, out=out).cpu()
        cache.bands.check(f"after step {s}")
    torch.cuda.synchronize()
    return dict(cache=cache, K=K, V=V, steps=steps, outs=outs, B=B, Hq=Hq, Hkv=Hkv, D=D,
                bits=bits, G=G, R=R, L=L, vqueue=vqueue)


def slot_bytes(run, b, h):
    """GPU bytes of one slot: (key parts [Lq/G, PART], value parts, k residual, v residual)."""
    c = run["cache"]
    lay = c.layout
    n_quant, n_resid = c.counts()
    G, D, Hkv = run["G"], run["D"], run["Hkv"]
    slot = b * Hkv + h
    buf = c.buffer
    base = slot * lay.slot_bytes
    nblk = n_quant // G
    kp = buf[base: base + nblk * lay.part_bytes].view(nblk, lay.part_bytes) if nblk else buf[:0].view(0, lay.part_bytes)
    vb = base + lay.blocks_per_slot * lay.part_bytes
    vp = buf[vb: vb + nblk * lay.part_bytes].view(nblk, lay.part_bytes) if nblk else buf[:0].view(0, lay.part_bytes)
    rk = buf[lay.k_resid_offset + slot * lay.resid_slot_bytes:][: n_resid * D * 2]
    if run.get("vqueue"):
        # the value queue: tokens [Lv, L) at ring rows position % R, in token order
        R = run["R"]
        L = n_quant + n_resid
        Lv = max(L - R, 0)
        ring = buf[lay.v_resid_offset + slot * lay.resid_slot_bytes:][: R * D * 2].view(R, D * 2)
        rv = ring[[t % R for t in range(Lv, L)]].reshape(-1) if L > Lv else ring[:0].reshape(-1)
    else:
        rv = buf[lay.v_resid_offset + slot * lay.resid_slot_bytes:][: n_resid * D * 2]
    return kp.cpu().numpy(), vp.cpu().numpy(), rk.cpu().numpy(), rv.cpu().numpy()


def oracle_slot(run, b, h, upto=None, on_step=None):
    """Replay slot (b, h) through the oracle; on_step(s, oracle_cache) after each append."""
    D, bits, G, R = run["D"], run["bits"], run["G"], run["R"]
    oc = (OracleCacheFifo if run.get("vqueue") else OracleCache)(1, 1, D, bits, G, R)
    oc.prefill(run["K"][b, h][None, None].cpu().numpy(), run["V"][b, h][None, None].cpu().numpy())
    n = len(run["steps"]) if upto is None else upto
    for s in range(n):
        _, k, v = run["steps"][s]
        oc.append(k[b, h][None, None].cpu().numpy(), v[b, h][None, None].cpu().numpy())
        if on_step is not None:
            on_step(s, oc)
    return oc


def check_slot_bytes(run, b, h, oc):
    """Bit-exact comparison of one slot's quantized blocks and residual rows."""
    bits, G = run["bits"], run["G"]
    kp, vp, rk, rv = slot_bytes(run, b, h)
    assert oc.n_quant == kp.shape[0] * G, (oc.n_quant, kp.shape)
    if oc.n_quant:
        ek = layout.pack_key_parts(oc.k_codes[0, 0], oc.k_s[0, 0], oc.k_z[0, 0], bits, G)
        vc, vs, vz = oc.v_codes[0, 0], oc.v_s[0, 0], oc.v_z[0, 0]
        if vc.shape[0] < oc.n_quant:
            # the value queue: tokens whose values are still queued read as zeros
            pad = oc.n_quant - vc.shape[0]
            vc = np.concatenate([vc, np.zeros((pad,) + vc.shape[1:], vc.dtype)])
            vs = np.concatenate([vs, np.zeros((pad,) + vs.shape[1:], vs.dtype)])
            vz = np.concatenate([vz, np.zeros((pad,) + vz.shape[1:], vz.dtype)])
        ev = layout.pack_value_parts(vc, vs, vz, bits, G)
        if not np.array_equal(kp, ek):
            bad = np.argwhere(kp != ek)[:5]
            raise AssertionError(f"key blocks differ at (block, byte) {bad.tolist()} in slot {(b, h)}")
        if not np.array_equal(vp, ev):
            bad = np.argwhere(vp != ev)[:5]
            raise AssertionError(f"value blocks differ at (block, byte) {bad.tolist()} in slot {(b, h)}")
    assert rk.tobytes() == oc.k_res[0, 0].tobytes(), f"key residual differs in slot {(b, h)}"
    assert rv.tobytes() == oc.v_res[0, 0].tobytes(), f"value residual differs in slot {(b, h)}"


def attention_ref(run, b, h, oc, s):
    """Oracle fp64 outputs of the query heads reading kv head h at step s: [rep][D]."""
    rep = run["Hq"] // run["Hkv"]
    q = run["steps"][s][0][b, h * rep:(h + 1) * rep].cpu().numpy()[None]
    o, _ = decode_attention(q, oc.keys_hat(), oc.values_hat())
    return o[0]


def assert_close(out, ref, what=""):
    out = np.asarray(out, np.float64)
    err = np.abs(out - ref)
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e} > {ATOL}"
    assert rel <= RTOL_L2, f"{what}: rel L2 err {rel:.3e} > {RTOL_L2}"
    return err.max(), rel


def check_slots(run, slots, decode_steps):
    """Replay each slot in the oracle; compare attention at decode steps and bytes at the end."""
    rep = run["Hq"] // run["Hkv"]
    worst = [0.0, 0.0]
    for (b, h) in slots:
        def on_step(s, oc):
            if s in decode_steps:
                ref = attention_ref(run, b, h, oc, s)
                got = run["outs"][s][b, h * rep:(h + 1) * rep].numpy()
                e, r = assert_close(got, ref, f"slot {(b, h)} step {s}")
                worst[0], worst[1] = max(worst[0], e), max(worst[1], r)
        oc = oracle_slot(run, b, h, on_step=on_step)
        check_slot_bytes(run, b, h, oc)
    return worst
