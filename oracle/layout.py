"""Packing of the oracle's logical cache into the library's byte layout.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages fix no storage format.  This module implements, independently of
the CUDA sources, the layout documented in the library header (include/kivi.h,
"Byte layout of the cache buffer"):

  * a slot's quantized tokens are in blocks of G tokens; each block has a key
    part and a value part of PART = (G/16)*TILE + 4*D bytes, TILE = 2*D*b;
  * a key part is G/16 code tiles, then the D channel steps (fp16), then the
    D channel zeros (fp16);
  * a value part is G/16 code tiles, then G/16 entry tiles: the steps of a
    code tile's 16 tokens as D/G rows of 16 fp16 (one row per channel group),
    then their zeros in the same form; inside a row, token t of the tile sits
    at position 4*((t % 8) // 2) + 2*(t // 8) + t % 2;
  * a code tile is 16 tokens x D channels in D*b/2 little-endian uint32
    words; lane l = 4g + i owns W = D*b/64 consecutive words.  Its code pairs
    are (k, r), k < D/16, r < 4:
      keys  : token g + 8(r%2), channels 16k + 2i + 8(r//2) (+1);
              class c = 2k + r//2, order h = r%2
      values: channel 16k + g + 8(r%2), tokens 2i + 8(r//2) (+1);
              class c = 2k + r%2, order h = r//2
    With P = 8/b, the pair lives in lane word c // P, byte h of each 16-bit
    half, bits b*(c % P) of that byte: the first code in the low half, the
    second in the high half.

Parity status: pinned (pack/unpack round trip covers every bit exactly once;
single-code tiles and single entries land on hand-computed words, bits and
bytes).
"""
from __future__ import annotations

import numpy as np


def sizes(D: int, b: int, G: int):
    """(TILE, PART) in bytes."""
    tile = 2 * D * b
    return tile, (G // 16) * tile + 4 * D


def _pair_coords(D: int, kind: str):
    """Coordinates of every code pair, indexed [lane 32][k D/16][r 4].

    Returns (tok0, ch0, tok1, ch1, cls, order): the first and second code's
    token and channel, the pair's class and order.
    """
    if kind not in ("key", "value"):
        raise ValueError(kind)
    lane, k, r = np.meshgrid(np.arange(32), np.arange(D // 16), np.arange(4), indexing="ij")
    g, i = lane // 4, lane % 4
    if kind == "key":
        tok0 = g + 8 * (r % 2)
        ch0 = 16 * k + 2 * i + 8 * (r // 2)
        tok1, ch1 = tok0, ch0 + 1
        cls, order = 2 * k + r // 2, r % 2
    else:
        ch0 = 16 * k + g + 8 * (r % 2)
        tok0 = 2 * i + 8 * (r // 2)
        tok1, ch1 = tok0 + 1, ch0
        cls, order = 2 * k + r % 2, r // 2
    return tok0, ch0, tok1, ch1, cls, order


def _placement(D: int, b: int, kind: str):
    """Per pair: (lane, lane word, bit of the first code) as flat int arrays,
    plus the pair coordinates flattened alike."""
    tok0, ch0, tok1, ch1, cls, order = _pair_coords(D, kind)
    P = 8 // b
    lane = np.broadcast_to(np.arange(32)[:, None, None], cls.shape)
    word = cls // P
    bit = 8 * order + b * (cls % P)
    flat = lambda a: np.ascontiguousarray(a).reshape(-1)
    return tuple(map(flat, (lane, word, bit, tok0, ch0, tok1, ch1)))


def pack_tiles(codes: np.ndarray, b: int, kind: str) -> np.ndarray:
    """codes uint8 [..., 16, D] -> uint32 [..., D*b/2] (one code tile each)."""
    *lead, T, D = codes.shape
    assert T == 16
    W = D * b // 64
    lane, word, bit, tok0, ch0, tok1, ch1 = _placement(D, b, kind)
    c0 = codes[..., tok0, ch0].astype(np.uint64)                 # [..., npairs]
    c1 = codes[..., tok1, ch1].astype(np.uint64)
    contrib = (c0 << bit.astype(np.uint64)) | (c1 << (bit + 16).astype(np.uint64))
    dest = lane * W + word                                       # each word receives 16/b pairs
    order = np.argsort(dest, kind="stable")
    per = 16 // b
    assert np.array_equal(dest[order].reshape(32 * W, per), np.repeat(np.arange(32 * W), per).reshape(-1, per))
    words = np.bitwise_or.reduce(contrib[..., order].reshape(*lead, 32 * W, per), axis=-1)
    return np.ascontiguousarray(words.astype("<u4"))


def unpack_tiles(words: np.ndarray, D: int, b: int, kind: str) -> np.ndarray:
    """Inverse of pack_tiles: uint32 [..., D*b/2] -> uint8 [..., 16, D]."""
    *lead, n = words.shape
    W = D * b // 64
    assert n == 32 * W
    lane, word, bit, tok0, ch0, tok1, ch1 = _placement(D, b, kind)
    w = words.astype(np.uint64)[..., lane * W + word]            # [..., npairs]
    mask = np.uint64((1 << b) - 1)
    out = np.zeros((*lead, 16, D), np.uint8)
    out[..., tok0, ch0] = ((w >> bit.astype(np.uint64)) & mask).astype(np.uint8)
    out[..., tok1, ch1] = ((w >> (bit + 16).astype(np.uint64)) & mask).astype(np.uint8)
    return out


def entry_position(t: int) -> int:
    """Position of token t (0..15 of a tile) inside a row of an entry tile."""
    return 4 * ((t % 8) // 2) + 2 * (t // 8) + t % 2


def pack_key_parts(codes: np.ndarray, s: np.ndarray, z: np.ndarray, b: int, G: int) -> np.ndarray:
    """Key parts of consecutive blocks.

    codes uint8 [nblk*G, D]; s, z fp16 [nblk, D]  ->  uint8 [nblk, PART].
    """
    T, D = codes.shape
    nblk = T // G
    tiles = pack_tiles(codes.reshape(nblk, G // 16, 16, D), b, "key")   # [nblk, G/16, D*b/2]
    tb = tiles.view(np.uint8).reshape(nblk, -1)
    sb = np.ascontiguousarray(s.astype("<f2")).view(np.uint8).reshape(nblk, -1)
    zb = np.ascontiguousarray(z.astype("<f2")).view(np.uint8).reshape(nblk, -1)
    return np.concatenate([tb, sb, zb], axis=1)


def _entry_tiles(s: np.ndarray, z: np.ndarray, G: int) -> np.ndarray:
    """Value (s, z) [nblk*G, D/G] -> entry tiles, uint8 [nblk, G/16 * 64*(D/G)]."""
    T, ngrp = s.shape
    nblk, ntile = T // G, G // 16
    perm = np.array([entry_position(t) for t in range(16)])
    rows_s = np.zeros((nblk, ntile, ngrp, 16), np.float16)
    rows_z = np.zeros((nblk, ntile, ngrp, 16), np.float16)
    st = s.reshape(nblk, ntile, 16, ngrp)
    zt = z.reshape(nblk, ntile, 16, ngrp)
    for t in range(16):
        rows_s[:, :, :, perm[t]] = st[:, :, t, :]
        rows_z[:, :, :, perm[t]] = zt[:, :, t, :]
    ent = np.concatenate([rows_s.reshape(nblk, ntile, -1), rows_z.reshape(nblk, ntile, -1)], axis=2)
    return np.ascontiguousarray(ent.astype("<f2")).view(np.uint8).reshape(nblk, -1)


def pack_value_parts(codes: np.ndarray, s: np.ndarray, z: np.ndarray, b: int, G: int) -> np.ndarray:
    """Value parts of consecutive blocks.

    codes uint8 [nblk*G, D]; s, z fp16 [nblk*G, D/G]  ->  uint8 [nblk, PART].
    """
    T, D = codes.shape
    nblk = T // G
    tiles = pack_tiles(codes.reshape(nblk, G // 16, 16, D), b, "value")
    tb = tiles.view(np.uint8).reshape(nblk, -1)
    return np.concatenate([tb, _entry_tiles(s, z, G)], axis=1)


def unpack_key_parts(parts: np.ndarray, D: int, b: int, G: int):
    """uint8 [nblk, PART] -> (codes [nblk*G, D], s [nblk, D], z [nblk, D])."""
    nblk = parts.shape[0]
    tile, _ = sizes(D, b, G)
    nt = G // 16
    words = np.ascontiguousarray(parts[:, : nt * tile]).view("<u4").reshape(nblk, nt, -1)
    codes = unpack_tiles(words, D, b, "key").reshape(nblk * G, D)
    ent = np.ascontiguousarray(parts[:, nt * tile:]).view("<f2").reshape(nblk, 2, D)
    return codes, ent[:, 0], ent[:, 1]


def unpack_value_parts(parts: np.ndarray, D: int, b: int, G: int):
    """uint8 [nblk, PART] -> (codes [nblk*G, D], s [nblk*G, D/G], z [nblk*G, D/G])."""
    nblk = parts.shape[0]
    tile, _ = sizes(D, b, G)
    nt, ngrp = G // 16, D // G
    words = np.ascontiguousarray(parts[:, : nt * tile]).view("<u4").reshape(nblk, nt, -1)
    codes = unpack_tiles(words, D, b, "value").reshape(nblk * G, D)
    ent = np.ascontiguousarray(parts[:, nt * tile:]).view("<f2").reshape(nblk, nt, 2, ngrp, 16)
    perm = np.array([entry_position(t) for t in range(16)])
    s = ent[:, :, 0][..., perm]                                  # [nblk, nt, ngrp, 16 tokens]
    z = ent[:, :, 1][..., perm]
    s = np.moveaxis(s, -1, -2).reshape(nblk * G, ngrp)
    z = np.moveaxis(z, -1, -2).reshape(nblk * G, ngrp)
    return codes, s, z
