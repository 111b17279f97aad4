"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Quantized blocks and residual rows are compared bit for bit; decode outputs
(fp16) against the oracle's fp64 attention over the same dequantized cache,
max |err| <= 4e-3 and relative L2 <= 1e-3.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU hosts too
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_kivi_kv_gb300.kivi import (KIVI_DECODE_CUDA_CORE, KIVI_DECODE_TENSOR_CORE,  # noqa: E402
                                    KIVI_ERR_CAPACITY, KIVI_ERR_STATE, KIVI_ERR_UNSUPPORTED, KiviCache,
                                    KiviError)

KERNELS = {"cuda_core": KIVI_DECODE_CUDA_CORE, "tensor_core": KIVI_DECODE_TENSOR_CORE}
from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV  # noqa: E402
from kivi_harness import check_slots, run_gpu  # noqa: E402


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_tiny_single_step(kernel):
    """B1 H1 D64, 2-bit, G32, R32: prefill 256 (224 quantized), append 1 (flush), decode."""
    run = run_gpu(1, 1, 1, 64, 2, 32, 32, L=256, n_app=1, seed=1000, decode_at={0},
                  outliers=FIXED_4_X20, sink=False, decode_kernel=KERNELS[kernel])
    assert run["cache"].counts() == (256, 1)
    check_slots(run, [(0, 0)], {0})


SMALL = [
    # B, Hq, Hkv, D, bits, G, R, L, n_app
    (2, 4, 4, 128, 2, 32, 128, 700, 12),      # ragged prompt, a flush after 4 appends
    (2, 8, 2, 128, 4, 128, 128, 1000, 10),    # grouped queries, 4-bit, G = R = 128
    (1, 4, 2, 64, 4, 64, 64, 300, 70),        # D64, 2 q heads per kv head, flushes
    (3, 2, 2, 64, 2, 32, 64, 0, 100),         # empty prompt: residual only, then flushes
    (2, 2, 2, 128, 2, 64, 128, 100, 5),       # prompt shorter than R: nothing quantized
    (1, 4, 1, 128, 2, 32, 32, 515, 40),       # 4 q heads per kv head, R = G
    (2, 2, 2, 128, 4, 32, 64, 161, 3),        # 4-bit with small groups
    (2, 4, 2, 128, 8, 32, 64, 333, 40),       # 8-bit, grouped queries, a flush
    (1, 2, 2, 64, 8, 64, 64, 200, 70),        # 8-bit D64 G64, flushes
]


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}D{c[3]}b{c[4]}G{c[5]}R{c[6]}L{c[7]}n{c[8]}" for c in SMALL])
def test_small_full_check(case, kernel):
    B, Hq, Hkv, D, bits, G, R, L, n = case
    steps = {0, n // 2, n - 1}
    run = run_gpu(B, Hq, Hkv, D, bits, G, R, L, n, seed=17 + sum(case), decode_at=steps,
                  decode_kernel=KERNELS[kernel])
    check_slots(run, [(b, h) for b in range(B) for h in range(Hkv)], steps)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}D{c[3]}b{c[4]}G{c[5]}R{c[6]}L{c[7]}n{c[8]}" for c in SMALL])
def test_fused_append_decode(case, kernel):
    """kivi_append_decode at every step (through residual fills and flushes)
    equals append + decode: outputs against the oracle at every step, then the
    cache bytes, including the residual rows the decode kernel stored."""
    B, Hq, Hkv, D, bits, G, R, L, n = case
    steps = set(range(n))
    run = run_gpu(B, Hq, Hkv, D, bits, G, R, L, n, seed=29 + sum(case), decode_at=steps,
                  decode_kernel=KERNELS[kernel], fused=True)
    check_slots(run, [(b, h) for b in range(B) for h in range(Hkv)], steps)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quantizer_near_ties(bits):
    """Groups whose elements sit exactly on half-steps (power-of-two steps make
    (x - z) / s = k + 1/2 exact, so rint breaks ties to even) or one fp16 ulp
    either side of them: the GPU codes must equal the oracle's fp32 formula."""
    L_b = (1 << bits) - 1
    B, H, D, G, R, L = 1, 1, 64, 32, 32, 32 * 9
    rng = np.random.default_rng(bits)
    def groups(n_groups, n):
        """n values per group: min 0, max L_b * s, then half-steps and their neighbours."""
        out = np.zeros((n_groups, n), np.float32)
        for gi in range(n_groups):
            # an fp16 power of two small enough that z + k*s stays exact in fp16
            s = np.float32(2.0 ** int(rng.integers(-6, 3) if bits < 8 else rng.integers(-9, -3)))
            z = np.float32(rng.choice([0.0, -1.0, 0.5, -3.25]))
            vals = [z, z + L_b * s]
            levels = range(L_b) if L_b < 16 else sorted(rng.choice(L_b, 10, replace=False))
            for k in levels:
                t = np.float16(z + (k + 0.5) * s)
                vals += [t, np.nextafter(t, np.float16(np.inf)), np.nextafter(t, np.float16(-np.inf))]
            while len(vals) < n:
                vals.append(z + s * np.float32(rng.integers(0, 4 * L_b + 1)) / 4)
            v = np.array(vals[:n], np.float32)
            v = np.clip(v, z, z + L_b * s)                          # keep min / max as set
            out[gi] = rng.permutation(v)
        return out.astype(np.float16)
    # keys: each channel over each block of G tokens is a group
    K = groups((L // G) * D, G).reshape(L // G, D, G).transpose(0, 2, 1).reshape(1, 1, L, D)
    # values: each token's G-channel groups
    V = groups(L * (D // G), G).reshape(1, 1, L, D)
    K = torch.from_numpy(np.ascontiguousarray(K)).cuda()
    V = torch.from_numpy(np.ascontiguousarray(V)).cuda()
    run = run_gpu(B, H, H, D, bits, G, R, L, 33, seed=11, decode_at={32}, prompt=(K, V))
    check_slots(run, [(0, 0)], {32})


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_crossings_near_zero(bits):
    """Groups with a step of 4-120 whose zero point puts a level's crossing
    z + (c - 1/2) s exactly at 0, where fp16 values are far denser than the
    crossing's rounding band (the threshold lies tens to hundreds of subnormal
    steps from 0), and whose other elements are consecutive fp16 values around
    both candidate sides: the GPU's level thresholds must give the oracle's codes
    bit for bit."""
    L_b = (1 << bits) - 1
    B, H, D, G, R, L = 1, 1, 64, 32, 32, 32 * 9
    rng = np.random.default_rng(100 + bits)
    def ordinal(h):
        b = int(np.float16(h).view(np.uint16))
        return -(b & 0x7FFF) if b & 0x8000 else b
    def from_ordinal(o):
        return np.uint16(o if o >= 0 else 0x8000 | -o).view(np.float16)
    def groups(n_groups, n):
        out = np.zeros((n_groups, n), np.float16)
        for gi in range(n_groups):
            c0 = int(rng.integers(1, L_b + 1))                     # the level whose crossing is at 0
            # a step of four significant bits, so z = -(c0 - 1/2) s and the max are exact fp16
            s16 = np.float16(2.0 ** int(rng.integers(2, 6)) * (1 + int(rng.integers(0, 8)) / 8))
            mn = np.float16(-(c0 - 0.5) * float(s16))
            mx = np.float16(float(mn) + L_b * float(s16))
            assert float(mn) == -(c0 - 0.5) * float(s16) and float(mx) - float(mn) == L_b * float(s16)
            # z + (c0 - 1/2) s is exactly 0; rn(x - z) stays at (c0 - 1/2) s for |x| under half
            # its fp32 ulp, so the threshold is about that far from 0 (its side set by the tie rule)
            half = float(np.spacing(np.float32((c0 - 0.5) * float(s16)))) / 2
            ot = ordinal(np.float16(half))
            ks = list(range(ot - 7, ot + 8)) + list(range(-ot - 7, -ot + 8))
            v = np.array([mn, mx] + [from_ordinal(k) for k in ks], np.float16)[:n]
            out[gi] = rng.permutation(v)
        return out
    K = groups((L // G) * D, G).reshape(L // G, D, G).transpose(0, 2, 1).reshape(1, 1, L, D)
    V = groups(L * (D // G), G).reshape(1, 1, L, D)
    K = torch.from_numpy(np.ascontiguousarray(K)).cuda()
    V = torch.from_numpy(np.ascontiguousarray(V)).cuda()
    run = run_gpu(B, H, H, D, bits, G, R, L, 33, seed=12, decode_at={32}, prompt=(K, V))
    check_slots(run, [(0, 0)], {32})


def test_degenerate_groups():
    """Constant key channels / value groups (step 0) and signed zeros: codes 0, zero +0."""
    B, H, D, G, R, L = 1, 2, 128, 32, 32, 160
    gen = torch.Generator().manual_seed(5)
    K = torch.randn(B, H, L, D, generator=gen)
    V = torch.randn(B, H, L, D, generator=gen)
    K[:, :, :, 5] = 1.5                       # a constant channel
    K[:, 0, 32:64, 9] = 0.0
    K[:, 0, 32:64:2, 9] = -0.0                # mixed signed zeros in one key group
    V[:, 1, 40, 32:64] = -2.25                # one constant value group
    V[:, 1, 41, :32] = -0.0
    K, V = K.half().cuda(), V.half().cuda()
    run = run_gpu(B, H, H, D, 2, G, R, L, 3, seed=3, decode_at={2}, prompt=(K, V))
    check_slots(run, [(0, 0), (0, 1)], {2})


def test_capacity_and_state_errors():
    c = KiviCache(1, 1, 1, 64, 2, 32, 32, max_tokens=40)
    K = torch.randn(1, 1, 41, 64, device="cuda").half()
    with pytest.raises(KiviError) as e:
        c.prefill(K, K)
    assert e.value.status == KIVI_ERR_CAPACITY
    c.prefill(K[:, :, :40].contiguous(), K[:, :, :40].contiguous())
    k = torch.randn(1, 1, 64, device="cuda").half()
    with pytest.raises(KiviError) as e:
        c.append(k, k)
    assert e.value.status == KIVI_ERR_CAPACITY
    assert c.counts() == (32, 8)


# ---- the full-size workloads, on sampled slots --------------------------------

def _slots(B, Hkv):
    return sorted({(0, 0), (B - 1, Hkv - 1), (B // 2, Hkv // 3)})


def test_llama2_7b_layer_fused_full_size():
    """The 7B-shaped layer decoded with kivi_append_decode at every one of 64 steps."""
    steps = set(range(64))
    run = run_gpu(8, 32, 32, 128, 2, 32, 128, 4096, 64, seed=1011, decode_at=steps,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, fused=True)
    check_slots(run, [(0, 0), (7, 31), (3, 17)], {0, 1, 31, 32, 63})


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_llama2_7b_layer_full_size(kernel):
    """B8 H32 D128, 2-bit G32 R128, prompt 4096 (sink + outliers), 64 decode steps."""
    steps = {0, 1, 31, 63}
    run = run_gpu(8, 32, 32, 128, 2, 32, 128, 4096, 64, seed=1001, decode_at=steps,
                  decode_kernel=KERNELS[kernel])
    assert run["cache"].counts() == (4096, 64)     # 3968 + one flush of 128; 64 appended
    check_slots(run, _slots(8, 32), steps)


def test_llama2_13b_layer_full_size():
    """One layer of the 40-layer B32 H40 D128 2-bit step: prompt 4096, append (flush), decode."""
    run = run_gpu(32, 40, 40, 128, 2, 32, 128, 4096, 1, seed=1002, decode_at={0})
    assert run["cache"].counts() == (4096, 1)
    check_slots(run, _slots(32, 40), {0})


def test_gqa_llama3_8b_full_size():
    """B64, 32 q heads on 8 kv heads, D128, 4-bit G128 R128, prompt 8192, append 1, decode."""
    run = run_gpu(64, 32, 8, 128, 4, 128, 128, 8192, 1, seed=1003, decode_at={0})
    assert run["cache"].counts() == (8192, 1)
    check_slots(run, _slots(64, 8), {0})


def test_long_context_streaming_full_size():
    """B2 H32 D128 2-bit G32 R128: prompt 131072, 512 appends (flush every 128)."""
    steps = {0, 1, 127, 128, 129, 255, 256, 383, 384, 385, 511}
    run = run_gpu(2, 32, 32, 128, 2, 32, 128, 131072, 512, seed=1004, decode_at=steps)
    assert run["cache"].counts() == (131072 + 384, 128)
    check_slots(run, [(0, 0), (1, 31)], steps)


COMBOS = [(D, bits, nq, G) for D in (64, 128) for bits in (2, 4, 8) for nq in (1, 2, 4)
          for G in (32, 64, 128) if G <= D]


@pytest.mark.parametrize("combo", COMBOS, ids=[f"D{c[0]}b{c[1]}nq{c[2]}G{c[3]}" for c in COMBOS])
def test_every_tensor_core_instantiation(combo):
    """Each (head_dim, bits, q-per-kv, G) kernel instance: ragged prompt, one
    flush, decode over quantized + residual tokens."""
    D, bits, nq, G = combo
    R = max(G, 64)
    L = 3 * G + R + 21
    run = run_gpu(2, 2 * nq, 2, D, bits, G, R, L, R - 20, seed=sum(combo), decode_at={0, R - 21},
                  decode_kernel=KIVI_DECODE_TENSOR_CORE)
    check_slots(run, [(0, 0), (1, 1)], {0, R - 21})


@pytest.mark.parametrize("fused", [False, True])
def test_many_short_slots(fused):
    """256 (batch, kv-head) slots of 200 + 40 tokens: each slot is shorter than a
    CTA's share, so the partition gives every slot a lead-in weight and CTAs
    cover several slot starts; sampled slots against the oracle at three steps."""
    steps = {0, 20, 39}
    run = run_gpu(16, 32, 16, 64, 2, 32, 64, 200, 40, seed=91, decode_at=steps,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, fused=fused)
    check_slots(run, [(0, 0), (3, 7), (7, 15), (8, 1), (12, 9), (15, 15)], steps)


# ---- value residual as a queue ([explainer] 3.2) ---------------------------------------------
VQ = [
    # B, Hq, Hkv, D, bits, G, R, L, n_app
    (2, 4, 4, 128, 2, 32, 128, 700, 140),     # ragged prompt, pops every step, key flushes
    (2, 8, 2, 128, 4, 128, 128, 1000, 10),    # grouped queries, 4-bit, G = R = 128
    (1, 4, 2, 64, 4, 64, 64, 300, 70),        # D64, flushes
    (3, 2, 2, 64, 2, 32, 64, 0, 100),         # empty prompt: the queue fills, then pops
    (2, 2, 2, 128, 2, 64, 128, 100, 5),       # prompt shorter than R: nothing quantized
    (1, 4, 1, 128, 2, 32, 32, 515, 40),       # R = G
    (2, 4, 2, 128, 8, 32, 64, 333, 40),       # 8-bit
]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", VQ, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}D{c[3]}b{c[4]}G{c[5]}R{c[6]}L{c[7]}n{c[8]}" for c in VQ])
def test_value_queue(case, fused):
    """The value queue: outputs at every step (keys flushing, values popping one
    token per append) and the cache bytes (blocks with queued values as zeros,
    the ring's rows) against the oracle's queue cache."""
    B, Hq, Hkv, D, bits, G, R, L, n = case
    steps = set(range(n))
    run = run_gpu(B, Hq, Hkv, D, bits, G, R, L, n, seed=53 + sum(case), decode_at=steps,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, fused=fused, vqueue=True)
    check_slots(run, [(b, h) for b in range(B) for h in range(Hkv)], steps)


@pytest.mark.parametrize("combo", COMBOS, ids=[f"D{c[0]}b{c[1]}nq{c[2]}G{c[3]}" for c in COMBOS])
def test_every_value_queue_instantiation(combo):
    """Each value-queue kernel instance: ragged prompt, a key flush, pops."""
    D, bits, nq, G = combo
    R = max(G, 64)
    L = 3 * G + R + 21
    steps = {0, 1, R - 22, R - 21}
    run = run_gpu(2, 2 * nq, 2, D, bits, G, R, L, R - 20, seed=sum(combo) + 5, decode_at=steps,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, fused=True, vqueue=True)
    check_slots(run, [(0, 0), (1, 1)], steps)


@pytest.mark.parametrize("max_ctas", [1, 5, 0])
def test_value_queue_mixed_calls(max_ctas):
    """Fused calls (whose decode kernel pops the oldest queued value) mixed with
    separate appends (whose own kernel pops it) and plain decodes right after
    a fused pop, on grids from one CTA (one warp pops for many slots) up."""
    B, Hq, Hkv, D, bits, G, R, L, n = 3, 8, 4, 128, 2, 32, 64, 500, 90
    steps = {s for s in range(n) if s % 5 != 4}
    fused = {s for s in range(n) if s % 3 != 2}
    run = run_gpu(B, Hq, Hkv, D, bits, G, R, L, n, seed=707 + max_ctas, decode_at=steps,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, fused=fused, vqueue=True, max_ctas=max_ctas)
    check_slots(run, [(b, h) for b in range(B) for h in range(Hkv)], steps)


def test_value_queue_pop_survives_a_failed_copy():
    """A fused call on a value-queue cache whose copy wait runs out (the fault
    hook: CTA 0, warp 0): the heads of the slot that warp covers come back NaN,
    every other head finite, and the cache is still exactly the oracle's, the
    pops included (each slot's pop runs before its warp's pair loop), so the
    following calls are correct."""
    from bit_kivi_kv_gb300.kivi import KIVI_FAULT_COPY_STALL, kivi_cache_set_fault
    from kivi_harness import check_slot_bytes, oracle_slot
    B, Hq, Hkv, D, bits, G, R, L, n = 2, 4, 4, 128, 2, 32, 64, 600, 6
    run = run_gpu(B, Hq, Hkv, D, bits, G, R, L, 0, seed=321, max_tokens=L + n,
                  decode_kernel=KIVI_DECODE_TENSOR_CORE, vqueue=True)
    cache, syn = run["cache"], SynthKV(B, Hq, Hkv, D, 321, device="cuda")
    for s in range(n):
        q, k, v = syn.step(s)
        run["steps"].append((q, k, v))
        if s == 2:
            kivi_cache_set_fault(cache.handle, KIVI_FAULT_COPY_STALL)
        run["outs"][s] = cache.append_decode(k, v, q, out=cache.bands.like(q))
        cache.bands.check(f"after step {s}")
    torch.cuda.synchronize()
    run["outs"] = {s: o.cpu() for s, o in run["outs"].items()}
    bad = run["outs"][2].float()
    assert torch.isnan(bad[0, 0]).all()                          # slot (0, 0): CTA 0's first slot
    assert torch.isfinite(bad[1]).all()
    # every byte of every slot, and the outputs of the calls after the failed one
    check_slots(run, [(b, h) for b in range(B) for h in range(Hkv)], {3, 4, 5})


def test_value_queue_llama2_7b_layer_full_size():
    """B8 H32 D128 2-bit G32 R128, prompt 4096, 64 fused appends with the value queue."""
    steps = {0, 1, 63}
    run = run_gpu(8, 32, 32, 128, 2, 32, 128, 4096, 64, seed=1001, decode_at=steps, fused=True, vqueue=True)
    check_slots(run, [(0, 0), (3, 17), (7, 31)], steps)


def test_value_queue_rules():
    c = KiviCache(1, 2, 2, 64, 2, 32, 64, 256)
    c.set_decode_kernel(KIVI_DECODE_CUDA_CORE)
    c.set_value_residual(1)
    syn_K = torch.zeros(1, 2, 100, 64, dtype=torch.float16, device="cuda")
    c.prefill(syn_K, syn_K)
    q = torch.zeros(1, 2, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(KiviError) as e:        # the queue is decoded by the tensor-core kernel only
        c.decode_attn(q)
    assert e.value.status == KIVI_ERR_UNSUPPORTED
    with pytest.raises(KiviError) as e:        # the mode is set on an empty cache
        c.set_value_residual(0)
    assert e.value.status == KIVI_ERR_STATE
    c.set_decode_kernel(KIVI_DECODE_TENSOR_CORE)
    out = c.decode_attn(q)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


def test_copy_wait_runs_out_marks_heads_and_context_stays_usable():
    """Failure detection without a fault: the test hook makes the first copy
    stage of CTA 0 wait for bytes that never come; its bounded wait gives up
    (about 2 s, twice), the heads of the slot CTA 0 covers come back NaN, every
    other head equals a clean call bit for bit, and the next call is clean."""
    from bit_kivi_kv_gb300.kivi import KIVI_FAULT_COPY_STALL, kivi_cache_set_fault
    B, H, D = 4, 8, 128
    syn = SynthKV(B, H, H, D, 99, device="cuda")
    K, V = syn.prompt(2048)
    c = KiviCache(B, H, H, D, 2, 32, 128, 2048)
    c.prefill(K, V)
    q = syn.step(0)[0]
    clean = c.decode_attn(q).clone()
    kivi_cache_set_fault(c.handle, KIVI_FAULT_COPY_STALL)
    bad = c.decode_attn(q)
    torch.cuda.synchronize()
    assert torch.isnan(bad[0, 0].float()).all()                 # slot (0, 0): CTA 0's only slot
    rest = torch.ones(B, H, dtype=torch.bool)
    rest[0, 0] = False
    assert torch.equal(bad[rest], clean[rest])
    again = c.decode_attn(q)
    torch.cuda.synchronize()
    assert torch.equal(again, clean)


def test_split_invariance():
    """The same decode call on grids of 1, 7, 64 CTAs and the default: a slot's
    split over CTAs changes, its arithmetic per token does not, so the outputs
    agree to fp32 summation order (within 1e-4, or one fp16 ulp of the value
    where that is larger)."""
    from bit_kivi_kv_gb300.kivi import kivi_cache_set_max_ctas
    B, H, D = 2, 8, 128
    syn = SynthKV(B, H, H, D, 7, device="cuda")
    K, V = syn.prompt(3000)
    c = KiviCache(B, H, H, D, 2, 32, 128, 3010)
    c.prefill(K, V)
    for s in range(5):
        _, k, v = syn.step(s)
        c.append(k, v)
    q = syn.step(5)[0]
    ref = c.decode_attn(q).float()
    for cap in (1, 7, 64):
        kivi_cache_set_max_ctas(c.handle, cap)
        out = c.decode_attn(q).float()
        ulp16 = torch.exp2(torch.floor(torch.log2(ref.abs().clamp(min=2.0 ** -14))) - 10)   # fp16 spacing at |ref|
        allowed = torch.clamp(ulp16, min=1e-4)
        assert torch.all((out - ref).abs() <= allowed), (cap, (out - ref).abs().max().item())
    kivi_cache_set_max_ctas(c.handle, 0)
    assert torch.equal(c.decode_attn(q).float(), ref)


def test_maximum_slot_count():
    """2047 x 32 = 65504 (batch, kv-head) slots, next to the 65535 limit the
    quantize grid's y dimension sets: prompt 96 (one quantized block, a full
    residual), 3 appends (the first flushes), decode; sampled slots against
    the oracle."""
    run = run_gpu(2047, 32, 32, 64, 2, 32, 64, 96, 3, seed=13, decode_at={2},
                  outliers=FIXED_4_X20, sink=False)
    assert run["cache"].counts() == (96, 3)
    check_slots(run, [(0, 0), (1023, 17), (2046, 31)], {2})
