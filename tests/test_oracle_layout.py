"""Pins for the oracle's packer and byte counts (no GPU)."""
import numpy as np
import pytest

from oracle import accounting, layout


@pytest.mark.parametrize("D,b", [(64, 2), (64, 4), (64, 8), (128, 2), (128, 4), (128, 8)])
@pytest.mark.parametrize("kind", ["key", "value"])
def test_round_trip_and_full_coverage(D, b, kind):
    rng = np.random.default_rng(D + b)
    codes = rng.integers(0, 1 << b, (5, 16, D)).astype(np.uint8)
    words = layout.pack_tiles(codes, b, kind)
    assert words.shape == (5, D * b // 2)
    assert np.array_equal(layout.unpack_tiles(words, D, b, kind), codes)
    full = np.full((16, D), (1 << b) - 1, np.uint8)
    assert np.all(layout.pack_tiles(full, b, kind) == 0xFFFFFFFF)      # every bit used
    # each element owns a disjoint field: single-code tiles set exactly b bits
    seen = np.zeros(D * b // 2 * 32, bool)
    for tok in range(16):
        for ch in range(D):
            one = np.zeros((16, D), np.uint8); one[tok, ch] = (1 << b) - 1
            bits = np.unpackbits(layout.pack_tiles(one, b, kind).view(np.uint8), bitorder="little")
            assert bits.sum() == b
            assert not np.any(seen & bits.astype(bool))
            seen |= bits.astype(bool)
    assert seen.all()


def test_single_code_positions(golden):
    for line in golden("layout_single_codes.txt"):
        kind, D, b, tok, ch, word, bit = line.split()
        D, b, tok, ch, word, bit = map(int, (D, b, tok, ch, word, bit))
        one = np.zeros((16, D), np.uint8); one[tok, ch] = 1
        w = layout.pack_tiles(one, b, kind)
        expect = np.zeros_like(w); expect[word] = 1 << bit
        assert np.array_equal(w, expect), line


def test_part_sizes_and_part_round_trip():
    assert layout.sizes(128, 2, 32) == (512, 1536)
    assert layout.sizes(128, 4, 128) == (1024, 8704)
    assert layout.sizes(64, 2, 32) == (256, 768)
    rng = np.random.default_rng(0)
    D, b, G, nblk = 128, 2, 32, 3
    kc = rng.integers(0, 4, (nblk * G, D)).astype(np.uint8)
    ks = rng.standard_normal((nblk, D)).astype(np.float16)
    kz = rng.standard_normal((nblk, D)).astype(np.float16)
    parts = layout.pack_key_parts(kc, ks, kz, b, G)
    assert parts.shape == (nblk, 1536)
    c2, s2, z2 = layout.unpack_key_parts(parts, D, b, G)
    assert np.array_equal(c2, kc) and s2.tobytes() == ks.tobytes() and z2.tobytes() == kz.tobytes()
    # steps of the D channels after the tiles, then their zeros
    assert parts[1, 1024 + 2 * 9: 1024 + 2 * 9 + 2].tobytes() == ks[1, 9].tobytes()
    assert parts[1, 1024 + 256 + 2 * 9: 1024 + 256 + 2 * 9 + 2].tobytes() == kz[1, 9].tobytes()
    vs = rng.standard_normal((nblk * G, D // G)).astype(np.float16)
    vz = rng.standard_normal((nblk * G, D // G)).astype(np.float16)
    vparts = layout.pack_value_parts(kc, vs, vz, b, G)
    c3, s3, z3 = layout.unpack_value_parts(vparts, D, b, G)
    assert np.array_equal(c3, kc) and s3.tobytes() == vs.tobytes() and z3.tobytes() == vz.tobytes()
    # block 2, token 5 (tile 0, row position 9), group 3
    off = 1024 + 2 * (3 * 16 + 9)
    assert vparts[2, off:off + 2].tobytes() == vs[2 * G + 5, 3].tobytes()
    assert vparts[2, off + 128:off + 130].tobytes() == vz[2 * G + 5, 3].tobytes()


def test_entry_positions(golden):
    """Single entries land on the hand-worked byte offsets."""
    assert [layout.entry_position(t) for t in range(16)] == [0, 1, 4, 5, 8, 9, 12, 13, 2, 3, 6, 7, 10, 11, 14, 15]
    for line in golden("layout_entries.txt"):
        kind, D, b, G, idx, grp, sb, zb = line.split()
        D, b, G, idx, sb, zb = map(int, (D, b, G, idx, sb, zb))
        s_mark, z_mark = np.float16(1.5), np.float16(-2.25)
        codes = np.zeros((G, D), np.uint8)
        if kind == "key":
            s = np.zeros((1, D), np.float16); z = np.zeros((1, D), np.float16)
            s[0, idx], z[0, idx] = s_mark, z_mark
            part = layout.pack_key_parts(codes, s, z, b, G)[0]
        else:
            s = np.zeros((G, D // G), np.float16); z = np.zeros((G, D // G), np.float16)
            s[idx, int(grp)], z[idx, int(grp)] = s_mark, z_mark
            part = layout.pack_value_parts(codes, s, z, b, G)[0]
        nz = np.flatnonzero(part)
        assert part[sb:sb + 2].tobytes() == s_mark.tobytes(), line
        assert part[zb:zb + 2].tobytes() == z_mark.tobytes(), line
        assert set(nz) <= {sb, sb + 1, zb, zb + 1}, line


def test_accounting(golden):
    lines = golden("accounting.txt")
    per_tok = int(lines[0].split()[1])
    assert accounting.fp16_kv_bytes(1, 1, 32, 4096) == per_tok
    assert abs(per_tok - 0.5 * 2**20) <= 0.05 * 2**20              # "about 0.5 MB"
    assert 19_000 <= (10 * 2**30) // per_tok <= 21_000                # "about 20,000 tokens in 10 GB"
    for line in lines[1:]:
        _, D, b, G, want = line.split()
        assert accounting.quantized_bytes_per_token(int(D), int(b), int(G)) == int(want)
    # a decode call of the 7B-shaped layer (B8 H32 D128, Lq 4096, r 1): 256*(4096*96+512)+2*8*32*128*2
    assert accounting.decode_call_bytes(8, 32, 32, 128, 2, 32, 4096, 1) == 256 * (4096 * 96 + 512) + 131072
