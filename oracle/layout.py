"""Packing of the oracle's logical cache into the library's byte layout.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages fix no storage format.  This module implements, independently of
the CUDA sources, the layout documented in the library header (include/kivi.h,
"Byte layout of the cache buffer"):

  * a slot's quantized tokens are in blocks of G tokens; each block has a key
    part and a value part of PART = (G/16)*TILE + 4*D bytes, TILE = 2*D*b;
  * a part is G/16 code tiles followed by fp16 (s, z) entries;
  * a code tile is 16 tokens x D channels in D*b/2 little-endian uint32
    words; lane l = 4g + i owns W = D*b/64 consecutive words; its pair p
    lives in word p // (16/b), slot u = p % (16/b), first code at bit b*u,
    second at bit 16 + b*u; with k = p // 4, r = p % 4:
      keys  : token g + 8(r%2), channels 16k + 2i + 8(r//2) (+1)
      values: channel 16k + g + 8(r%2), tokens 2i + 8(r//2) (+1)

Parity status: pinned (pack/unpack round trip covers every bit exactly once;
single-code tiles land on the hand-computed word and bit).
"""
from __future__ import annotations

import numpy as np


def sizes(D: int, b: int, G: int):
    """(TILE, PART) in bytes."""
    tile = 2 * D * b
    return tile, (G // 16) * tile + 4 * D


def _maps(D: int, b: int, kind: str):
    """Index maps over [lane 32][pair D/4]: (tok0, ch0, tok1, ch1, shift)."""
    if kind not in ("key", "value"):
        raise ValueError(kind)
    l, p = np.meshgrid(np.arange(32), np.arange(D // 4), indexing="ij")
    g, i = l // 4, l % 4
    k, r = p // 4, p % 4
    shift = b * (p % (16 // b))
    if kind == "key":
        tok0 = g + 8 * (r % 2)
        tok1 = tok0
        ch0 = 16 * k + 2 * i + 8 * (r // 2)
        ch1 = ch0 + 1
    else:
        ch0 = 16 * k + g + 8 * (r % 2)
        ch1 = ch0
        tok0 = 2 * i + 8 * (r // 2)
        tok1 = tok0 + 1
    return tok0, ch0, tok1, ch1, shift


def pack_tiles(codes: np.ndarray, b: int, kind: str) -> np.ndarray:
    """codes uint8 [..., 16, D] -> uint32 [..., D*b/2] (one code tile each)."""
    *lead, T, D = codes.shape
    assert T == 16
    tok0, ch0, tok1, ch1, shift = _maps(D, b, kind)
    c0 = codes[..., tok0, ch0].astype(np.uint32)        # [..., 32, D/4]
    c1 = codes[..., tok1, ch1].astype(np.uint32)
    contrib = (c0 << shift.astype(np.uint32)) | (c1 << (shift + 16).astype(np.uint32))
    W, per = D * b // 64, 16 // b
    contrib = contrib.reshape(*lead, 32, W, per)
    words = np.bitwise_or.reduce(contrib, axis=-1)     # [..., 32, W]
    return np.ascontiguousarray(words.reshape(*lead, 32 * W).astype("<u4"))


def unpack_tiles(words: np.ndarray, D: int, b: int, kind: str) -> np.ndarray:
    """Inverse of pack_tiles: uint32 [..., D*b/2] -> uint8 [..., 16, D]."""
    *lead, n = words.shape
    W, per = D * b // 64, 16 // b
    assert n == 32 * W
    tok0, ch0, tok1, ch1, shift = _maps(D, b, kind)
    w = words.astype(np.uint32).reshape(*lead, 32, W, 1)
    w = np.broadcast_to(w, (*lead, 32, W, per)).reshape(*lead, 32, W * per)   # [..., 32, D/4]
    mask = np.uint32((1 << b) - 1)
    v0 = ((w >> shift.astype(np.uint32)) & mask).astype(np.uint8)
    v1 = ((w >> (shift + 16).astype(np.uint32)) & mask).astype(np.uint8)
    out = np.zeros((*lead, 16, D), np.uint8)
    out[..., tok0, ch0] = v0
    out[..., tok1, ch1] = v1
    return out


def _entries(s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """(s, z) fp16 pairs as bytes, s first."""
    return np.stack([s, z], axis=-1).astype("<f2").view(np.uint8)


def pack_key_parts(codes: np.ndarray, s: np.ndarray, z: np.ndarray, b: int, G: int) -> np.ndarray:
    """Key parts of consecutive blocks.

    codes uint8 [nblk*G, D]; s, z fp16 [nblk, D]  ->  uint8 [nblk, PART].
    """
    T, D = codes.shape
    nblk = T // G
    tiles = pack_tiles(codes.reshape(nblk, G // 16, 16, D), b, "key")   # [nblk, G/16, D*b/2]
    tb = tiles.view(np.uint8).reshape(nblk, -1)
    ent = _entries(s, z).reshape(nblk, -1)
    return np.concatenate([tb, ent], axis=1)


def pack_value_parts(codes: np.ndarray, s: np.ndarray, z: np.ndarray, b: int, G: int) -> np.ndarray:
    """Value parts of consecutive blocks.

    codes uint8 [nblk*G, D]; s, z fp16 [nblk*G, D/G]  ->  uint8 [nblk, PART].
    """
    T, D = codes.shape
    nblk = T // G
    tiles = pack_tiles(codes.reshape(nblk, G // 16, 16, D), b, "value")
    tb = tiles.view(np.uint8).reshape(nblk, -1)
    ent = _entries(s, z).reshape(nblk, -1)      # token-major, group-minor
    return np.concatenate([tb, ent], axis=1)


def unpack_key_parts(parts: np.ndarray, D: int, b: int, G: int):
    """uint8 [nblk, PART] -> (codes [nblk*G, D], s [nblk, D], z [nblk, D])."""
    nblk = parts.shape[0]
    tile, _ = sizes(D, b, G)
    nt = G // 16
    words = np.ascontiguousarray(parts[:, : nt * tile]).view("<u4").reshape(nblk, nt, -1)
    codes = unpack_tiles(words, D, b, "key").reshape(nblk * G, D)
    ent = np.ascontiguousarray(parts[:, nt * tile:]).view("<f2").reshape(nblk, D, 2)
    return codes, ent[..., 0], ent[..., 1]


def unpack_value_parts(parts: np.ndarray, D: int, b: int, G: int):
    """uint8 [nblk, PART] -> (codes [nblk*G, D], s [nblk*G, D/G], z [nblk*G, D/G])."""
    nblk = parts.shape[0]
    tile, _ = sizes(D, b, G)
    nt = G // 16
    words = np.ascontiguousarray(parts[:, : nt * tile]).view("<u4").reshape(nblk, nt, -1)
    codes = unpack_tiles(words, D, b, "value").reshape(nblk * G, D)
    ent = np.ascontiguousarray(parts[:, nt * tile:]).view("<f2").reshape(nblk * G, D // G, 2)
    return codes, ent[..., 0], ent[..., 1]
