"""GPU parity helpers for the paged cache: drive a serving-like schedule of
sequences (adds with ragged prompts, append + decode over changing subsets,
decode-only calls, releases whose pages are reused) through the C ABI, then
replay every sequence with the CPU oracle and compare outputs and bytes."""
from __future__ import annotations

import numpy as np
import torch

from bit_kivi_kv_gb300.synth import RANGE_2_6_X10_50, SynthKV
from guards import GuardedPagedCache
from kivi_harness import assert_close
from oracle import layout
from oracle.attention import decode_attention
from oracle.cache import OracleCache


class PagedRun:
    def __init__(self, Hq, Hkv, D, bits, G, R, max_seqs, max_blocks, n_pages, seed, outliers=RANGE_2_6_X10_50,
                 check_heads=None):
        self.Hq, self.Hkv, self.D, self.bits, self.G, self.R = Hq, Hkv, D, bits, G, R
        self.max_blocks, self.seed, self.outliers = max_blocks, seed, outliers
        self.check_heads = list(range(Hkv)) if check_heads is None else list(check_heads)
        # pool, workspace and outputs between guard bands, checked after every call
        self.cache = GuardedPagedCache(max_seqs, Hq, Hkv, D, bits, G, R, max_blocks, n_pages)
        self.live = {}       # seq id -> record
        self.n_made = 0
        self.checked = 0     # sequences checked (released or at the end)
        self.worst = [0.0, 0.0]

    def add(self, L):
        syn = SynthKV(1, self.Hq, self.Hkv, self.D, self.seed * 7919 + self.n_made, outliers=self.outliers,
                      sink=True, device="cuda")
        self.n_made += 1
        K, V = syn.prompt(L)
        K, V = K[0].contiguous(), V[0].contiguous()
        s = self.cache.add(K, V)
        self.cache.bands.check(f"after adding a prompt of {L} tokens")
        assert s not in self.live
        self.live[s] = dict(syn=syn, K=K.cpu().numpy(), V=V.cpu().numpy(), events=[], n_steps=0)
        return s

    def step(self, seqs, append=True):
        """One call over seqs (in this order): append + decode, or decode only."""
        qs, ks, vs = [], [], []
        for s in seqs:
            rec = self.live[s]
            q, k, v = rec["syn"].step(rec["n_steps"])
            rec["n_steps"] += 1
            qs.append(q[0]); ks.append(k[0]); vs.append(v[0])
        Q = torch.stack(qs).contiguous()
        Kn = torch.stack(ks).contiguous() if append else None
        Vn = torch.stack(vs).contiguous() if append else None
        out = self.cache.append_decode(seqs, Kn, Vn, Q, out=self.cache.bands.like(Q))
        self.cache.bands.check(f"after the call over {list(seqs)}")
        out = out.cpu().numpy()
        for i, s in enumerate(seqs):
            ev = self.live[s]["events"]
            if append:
                ev.append(("append", ks[i].cpu().numpy(), vs[i].cpu().numpy()))
            ev.append(("decode", qs[i].cpu().numpy(), out[i]))
        return out

    def release(self, s):
        torch.cuda.synchronize()
        self.check(s)
        self.cache.release(s)
        del self.live[s]

    def check_all(self):
        torch.cuda.synchronize()
        for s in sorted(self.live):
            self.check(s)
        return self.worst

    # -- oracle replay of one sequence --------------------------------------------
    def check(self, s):
        rec = self.live[s]
        rep = self.Hq // self.Hkv
        D, G, R, bits = self.D, self.G, self.R, self.bits
        n_quant, n_resid = self.cache.counts(s)
        pages = self.cache.pages(s)
        assert len(pages) * G == n_quant, (s, len(pages), n_quant)
        lay = self.cache.layout
        buf = self.cache.buffer
        table = buf[lay.table_offset + s * self.max_blocks * 4:][: len(pages) * 4].cpu().numpy().view(np.int32)
        assert table.tolist() == pages, f"block table row of sequence {s}"
        for h in self.check_heads:
            oc = OracleCache(1, 1, D, bits, G, R)
            oc.prefill(rec["K"][h][None, None], rec["V"][h][None, None])
            for ev in rec["events"]:
                if ev[0] == "append":
                    oc.append(ev[1][h][None, None], ev[2][h][None, None])
                else:
                    q = ev[1][h * rep:(h + 1) * rep][None]
                    ref, _ = decode_attention(q, oc.keys_hat(), oc.values_hat())
                    e, r = assert_close(ev[2][h * rep:(h + 1) * rep], ref[0], f"sequence {s} head {h}")
                    self.worst[0], self.worst[1] = max(self.worst[0], e), max(self.worst[1], r)
            assert oc.n_quant == n_quant and oc.n_resid == n_resid, (s, oc.n_quant, oc.n_resid, n_quant, n_resid)
            # blocks: page p holds head h's key part at (p*Hkv + h)*2*PART, the value part after it
            if n_quant:
                kp = np.stack([buf[(p * self.Hkv + h) * 2 * lay.part_bytes:][: lay.part_bytes].cpu().numpy()
                               for p in pages])
                vp = np.stack([buf[((p * self.Hkv + h) * 2 + 1) * lay.part_bytes:][: lay.part_bytes].cpu().numpy()
                               for p in pages])
                ek = layout.pack_key_parts(oc.k_codes[0, 0], oc.k_s[0, 0], oc.k_z[0, 0], bits, G)
                ev_ = layout.pack_value_parts(oc.v_codes[0, 0], oc.v_s[0, 0], oc.v_z[0, 0], bits, G)
                if not np.array_equal(kp, ek):
                    bad = np.argwhere(kp != ek)[:5]
                    raise AssertionError(f"key blocks of sequence {s} head {h} differ at {bad.tolist()}")
                if not np.array_equal(vp, ev_):
                    bad = np.argwhere(vp != ev_)[:5]
                    raise AssertionError(f"value blocks of sequence {s} head {h} differ at {bad.tolist()}")
            rows = (s * self.Hkv + h) * R * D * 2
            rk = buf[lay.k_resid_offset + rows:][: n_resid * D * 2].cpu().numpy()
            rv = buf[lay.v_resid_offset + rows:][: n_resid * D * 2].cpu().numpy()
            assert rk.tobytes() == oc.k_res[0, 0].tobytes(), f"key residual of sequence {s} head {h}"
            assert rv.tobytes() == oc.v_res[0, 0].tobytes(), f"value residual of sequence {s} head {h}"
        self.checked += 1
