"""GPU parity of the paged cache (ragged sequences, block tables) against the
CPU oracle: every decode output of every call, then each sequence's pages,
block-table row and residual rows bit for bit (checked before a sequence is
released, since its pages are then reused)."""
import random

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU hosts too
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_kivi_kv_gb300.kivi import (KIVI_ERR_CAPACITY, KIVI_ERR_STATE, KiviCache,  # noqa: E402
                                    KiviError, KiviPagedCache)
from bit_kivi_kv_gb300.synth import SynthKV  # noqa: E402
from paged_harness import PagedRun  # noqa: E402


def serve(run, lengths, n_steps, rng, churn_at=(), decode_only_at=(), new_lengths=()):
    """Add sequences with the given prompt lengths, then n_steps calls over
    random subsets in random order; at each step in churn_at one sequence is
    released and a new one added (its pages come from the released ones)."""
    for L in lengths:
        run.add(L)
    new_lengths = list(new_lengths)
    for t in range(n_steps):
        if t in churn_at and run.live:
            run.release(rng.choice(sorted(run.live)))
            run.add(new_lengths.pop(0) if new_lengths else rng.randrange(0, 400))
        live = sorted(run.live)
        k = rng.randint(1, len(live))
        seqs = rng.sample(live, k)
        if t in decode_only_at:
            seqs = [s for s in seqs if sum(run.cache.counts(s)) > 0] or seqs[:0]
            if seqs:
                run.step(seqs, append=False)
            continue
        run.step(seqs)
    return run.check_all()


def test_paged_ragged_schedule():
    """Eight sequences of ragged prompts (empty, 1 token, around R, several
    blocks), 70 calls over random subsets with flushes at different steps,
    decode-only calls, and three release + add churns reusing pages."""
    rng = random.Random(5)
    run = PagedRun(Hq=4, Hkv=2, D=128, bits=2, G=32, R=64, max_seqs=10, max_blocks=24, n_pages=120, seed=1)
    serve(run, [0, 1, 63, 64, 65, 200, 333, 700], 70, rng, churn_at={15, 30, 50}, decode_only_at={10, 40},
          new_lengths=[97, 0, 511])
    assert run.checked >= 11


COMBOS = [(D, bits, nq, G) for D in (64, 128) for bits in (2, 4, 8) for nq in (1, 2, 4)
          for G in (32, 64, 128) if G <= D]


@pytest.mark.parametrize("combo", COMBOS, ids=[f"D{c[0]}b{c[1]}nq{c[2]}G{c[3]}" for c in COMBOS])
def test_every_paged_instantiation(combo):
    """Each paged kernel instance: three ragged sequences, a flush of one of
    them, a release + add, decode over quantized + residual tokens."""
    D, bits, nq, G = combo
    R = max(G, 64)
    rng = random.Random(sum(combo))
    run = PagedRun(Hq=2 * nq, Hkv=2, D=D, bits=bits, G=G, R=R, max_seqs=4, max_blocks=12, n_pages=30,
                   seed=sum(combo))
    serve(run, [3 * G + R + 5, R // 2, G + R], 24, rng, churn_at={12}, new_lengths=[2 * G + R])


@pytest.mark.parametrize("shape", [(128, 2, 32, 6000, 4), (64, 4, 64, 9500, 4), (128, 4, 128, 20000, 2)],
                         ids=["D128b2G32", "D64b4G64", "D128b4G128nq1"])
def test_paged_one_cta_grid_long_segments(shape):
    """A one-CTA grid: each warp's share of a sequence runs past the 128 block
    offsets a warp caches per segment, so the segment runs in parts with the
    cache refilled between them (G 128: four tile pairs a block; one query head
    per kv head: key fragments read from the warp's table)."""
    from bit_kivi_kv_gb300.kivi import kivi_paged_set_max_ctas
    D, bits, G, L, Hq = shape
    nb = (L + 40) // G + 2
    run = PagedRun(Hq=Hq, Hkv=2, D=D, bits=bits, G=G, R=2 * G, max_seqs=2, max_blocks=nb, n_pages=2 * nb, seed=11)
    kivi_paged_set_max_ctas(run.cache.handle, 1)
    a, b = run.add(L), run.add(L - 700)
    for t in range(12):
        run.step([a, b] if t % 2 == 0 else [b, a])
    run.check_all()


def test_paged_equals_dense_for_equal_lengths():
    """Sequences of equal length, listed in slot order, give the dense cache's
    outputs exactly: the weight partition and every kernel's arithmetic are the
    same, only the block addresses differ.  Listed in another order the split
    points of a sequence move, so the outputs agree within the tolerance."""
    from kivi_harness import ATOL
    B, Hq, Hkv, D, bits, G, R, L, n = 4, 8, 8, 128, 2, 32, 128, 700, 40
    syn = SynthKV(B, Hq, Hkv, D, 77, device="cuda")
    K, V = syn.prompt(L)
    dense = KiviCache(B, Hq, Hkv, D, bits, G, R, L + n + 1)
    dense.prefill(K, V)
    paged = KiviPagedCache(B, Hq, Hkv, D, bits, G, R, (L + n) // G + 1, 4 * ((L + n) // G + 1))
    seqs = [paged.add(K[b].contiguous(), V[b].contiguous()) for b in range(B)]
    for s in range(n):
        q, k, v = syn.step(s)
        od = dense.append_decode(k, v, q)
        op = paged.append_decode(seqs, k, v, q)
        assert torch.equal(op, od), f"step {s}"
    perm = [2, 0, 3, 1]
    q, k, v = syn.step(n)
    od = dense.append_decode(k, v, q)
    op = paged.append_decode([seqs[b] for b in perm], k[perm].contiguous(), v[perm].contiguous(),
                             q[perm].contiguous())
    assert (op.float() - od[perm].float()).abs().max().item() <= ATOL


def test_paged_capacity_errors_leave_state_unchanged():
    """A flush that needs more free pages than the pool has, a full sequence,
    and a decode-only call on an empty sequence are refused before any launch."""
    D, G, R = 64, 32, 32
    c = KiviPagedCache(3, 2, 2, D, 2, G, R, 3, 4)
    syn = SynthKV(1, 2, 2, D, 3, device="cuda")
    K, V = syn.prompt(96)                      # Lq = 64: two pages
    a = c.add(K[0].contiguous(), V[0].contiguous())
    K2, V2 = syn.prompt(64)                    # Lq = 32: one page
    b = c.add(K2[0].contiguous(), V2[0].contiguous())
    e = c.add(K2[0][:, :0].contiguous(), V2[0][:, :0].contiguous())
    assert c.free() == (1, 0)
    q, k, v = syn.step(0)
    qq = q.repeat(2, 1, 1).contiguous()
    kk = k.repeat(2, 1, 1).contiguous()
    vv = v.repeat(2, 1, 1).contiguous()
    # a and b both hold R residual tokens: flushing both needs 2 pages, 1 is free
    with pytest.raises(KiviError) as err:
        c.append_decode([a, b], kk, vv, qq)
    assert err.value.status == KIVI_ERR_CAPACITY
    assert c.counts(a) == (64, 32) and c.counts(b) == (32, 32) and c.free() == (1, 0)
    with pytest.raises(KiviError) as err:     # decode only on the empty sequence
        c.append_decode([e], None, None, q.contiguous())
    assert err.value.status == KIVI_ERR_STATE
    c.append_decode([b], k.contiguous(), v.contiguous(), q.contiguous())   # b flushes into the last page
    assert c.counts(b) == (64, 1) and c.free() == (0, 0)
    # a's flush needs a third page and none is free
    with pytest.raises(KiviError) as err:
        c.append_decode([a], k.contiguous(), v.contiguous(), q.contiguous())
    assert err.value.status == KIVI_ERR_CAPACITY
    c.release(b)
    assert c.free() == (2, 1)
    out = c.append_decode([a], k.contiguous(), v.contiguous(), q.contiguous())
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert c.counts(a) == (96, 1) and c.free() == (1, 1)


def test_paged_7b_shape_ragged_full_size():
    """Llama-2-7B layer shape (H32 D128, 2-bit, G32, R128) with 8 sequences of
    ragged prompts between 700 and 8000 tokens, 40 calls (each sequence
    flushes at its own step); every output and byte of kv heads 0, 17 and 31
    checked, the block tables of all."""
    rng = random.Random(11)
    run = PagedRun(Hq=32, Hkv=32, D=128, bits=2, G=32, R=128, max_seqs=8, max_blocks=260, n_pages=8 * 260,
                   seed=3, check_heads=[0, 17, 31])
    lengths = [700, 8000, 1234, 4096, 3000, 129, 6001, 2500]
    for L in lengths:
        run.add(L)
    for t in range(40):
        run.step(list(range(8)) if t % 3 else rng.sample(range(8), 5))
    run.check_all()
