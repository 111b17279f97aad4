"""Guard bands around the library's device buffers, in place of a memory checker.

Every buffer the library writes (the cache buffer or page pool, the decode
workspace, the decode outputs) is placed between two 4 KiB bands filled with a
fixed byte pattern.  A kernel that writes past either end of its buffer
changes a band; the harness checks the bands after every call.
"""
from __future__ import annotations

import torch

from bit_kivi_kv_gb300.kivi import KiviCache, KiviPagedCache

GUARD = 4096    # bytes on each side; keeps the 256-byte alignment of torch's allocations


def _pattern(n, device, salt):
    g = torch.Generator(device="cpu").manual_seed(0x5EED + salt)
    return torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8).to(device)


class Banded:
    """A list of (padded tensor, band pattern) pairs with one check over all of them."""

    def __init__(self):
        self.items = []

    def bytes(self, nbytes, device):
        """A uint8 view of nbytes between two bands."""
        pad = torch.empty(nbytes + 2 * GUARD, dtype=torch.uint8, device=device)
        pat = _pattern(2 * GUARD, device, len(self.items))
        pad[:GUARD] = pat[:GUARD]
        pad[GUARD + nbytes:] = pat[GUARD:]
        self.items.append((pad, pat, nbytes))
        return pad[GUARD:GUARD + nbytes]

    def like(self, t):
        """An uninitialized tensor shaped like t, between two bands."""
        n = t.numel() * t.element_size()
        return self.bytes(n, t.device).view(t.dtype).view(t.shape)

    def check(self, what=""):
        for i, (pad, pat, n) in enumerate(self.items):
            lo, hi = pad[:GUARD], pad[GUARD + n:]
            if not (torch.equal(lo, pat[:GUARD]) and torch.equal(hi, pat[GUARD:])):
                bad_lo = int((lo != pat[:GUARD]).sum())
                bad_hi = int((hi != pat[GUARD:]).sum())
                raise AssertionError(f"guard band of buffer {i} ({n} bytes) overwritten {what}: "
                                     f"{bad_lo} bytes below, {bad_hi} bytes above")


class GuardedCache(KiviCache):
    """KiviCache whose buffer and workspace sit between guard bands."""

    def __init__(self, *args, **kw):
        self.bands = Banded()
        super().__init__(*args, **kw)

    def _alloc(self, nbytes, device):
        return self.bands.bytes(nbytes, device)


class GuardedPagedCache(KiviPagedCache):
    """KiviPagedCache whose page pool (with residual rows and block table) and
    workspace sit between guard bands."""

    def __init__(self, *args, **kw):
        self.bands = Banded()
        super().__init__(*args, **kw)

    def _alloc(self, nbytes, device):
        return self.bands.bytes(nbytes, device)
