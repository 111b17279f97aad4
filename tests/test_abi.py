"""The C-ABI library builds, loads and exports every declared symbol; host-only
argument checks behave as include/kivi.h states (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    from bit_kivi_kv_gb300 import build
    build.build()
    from bit_kivi_kv_gb300 import kivi
    return kivi


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(kivi_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(K):
    names = _declared()
    assert len(names) >= 12, names
    lib = ctypes.CDLL(K._LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_config_validation(K):
    ok = K.make_config(8, 32, 32, 128, 2, 32, 128, 4160)
    assert K.kivi_cache_bytes(ok) > 0
    bad = [K.make_config(8, 32, 32, 96, 2, 32, 128, 4160),     # head_dim
           K.make_config(8, 32, 32, 128, 3, 32, 128, 4160),    # bits
           K.make_config(8, 32, 32, 128, 2, 48, 96, 4160),     # group
           K.make_config(8, 32, 32, 128, 2, 32, 100, 4160),    # residual % group
           K.make_config(8, 32, 32, 64, 2, 128, 128, 4160),    # head_dim % group
           K.make_config(8, 24, 16, 128, 2, 32, 128, 4160),    # heads ratio
           K.make_config(8, 32, 32, 128, 2, 32, 128, 0)]       # max_tokens
    for cfg in bad:
        assert K.kivi_cache_bytes(cfg) == 0
        assert K.kivi_last_error_string()
        assert K.kivi_decode_workspace_bytes(cfg) == 0


def test_layout_closed_forms(K):
    cfg = K.make_config(8, 32, 32, 128, 2, 32, 128, 4160)
    lay = K.kivi_cache_layout(cfg)
    assert (lay.tile_bytes, lay.part_bytes, lay.blocks_per_slot) == (512, 1536, 130)
    assert lay.slot_bytes == 2 * 130 * 1536
    assert lay.k_resid_offset % 256 == 0 and lay.v_resid_offset % 256 == 0
    assert lay.k_resid_offset >= 256 * lay.slot_bytes
    assert lay.v_resid_offset >= lay.k_resid_offset + 256 * 128 * 128 * 2
    assert lay.total_bytes == K.kivi_cache_bytes(cfg)


def test_host_side_checks_without_gpu(K):
    cfg = K.make_config(1, 1, 1, 64, 2, 32, 32, 64)
    n = K.kivi_cache_bytes(cfg)
    fake = 1 << 20                                  # never dereferenced by host-only calls
    with pytest.raises(K.KiviError) as e:
        K.kivi_cache_create(cfg, fake + 16, n)
    assert e.value.status == K.KIVI_ERR_INVALID_ARG
    with pytest.raises(K.KiviError) as e:
        K.kivi_cache_create(cfg, fake, n - 1)
    assert e.value.status == K.KIVI_ERR_CAPACITY
    h = K.kivi_cache_create(cfg, fake, n)
    try:
        assert K.kivi_cache_counts(h) == (0, 0)
        with pytest.raises(K.KiviError) as e:       # decode on an empty cache
            K.kivi_decode_attn(h, fake, fake, 0.0, fake, 1 << 30, 0)
        assert e.value.status == K.KIVI_ERR_STATE
        with pytest.raises(K.KiviError) as e:       # prompt longer than max_tokens
            K.kivi_prefill(h, fake, fake, 65, 0)
        assert e.value.status == K.KIVI_ERR_CAPACITY
        K.kivi_prefill(h, fake, fake, 0, 0)        # empty prompt: no work, no launch
        assert K.kivi_cache_counts(h) == (0, 0)
        with pytest.raises(K.KiviError) as e:
            K.kivi_append(h, 0, fake, 0)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        with pytest.raises(K.KiviError) as e:
            K.kivi_append(h, fake + 8, fake, 0)     # misaligned
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        ws_need = K.kivi_decode_workspace_bytes(cfg)
        # fused append + decode: argument checks run before anything is launched
        for args, status in [((0, fake, fake, fake, 0.0, fake, ws_need), K.KIVI_ERR_INVALID_ARG),
                             ((fake + 8, fake, fake, fake, 0.0, fake, ws_need), K.KIVI_ERR_INVALID_ARG),
                             ((fake, fake, 0, fake, 0.0, fake, ws_need), K.KIVI_ERR_INVALID_ARG),
                             ((fake, fake, fake, fake, 0.0, fake + 64, ws_need), K.KIVI_ERR_INVALID_ARG),
                             ((fake, fake, fake, fake, float("nan"), fake, ws_need), K.KIVI_ERR_INVALID_ARG),
                             ((fake, fake, fake, fake, 0.0, fake, ws_need - 1), K.KIVI_ERR_CAPACITY)]:
            with pytest.raises(K.KiviError) as e:
                K.kivi_append_decode(h, *args, 0)
            assert e.value.status == status, (args, e.value.status)
        assert K.kivi_cache_counts(h) == (0, 0)
        K.kivi_cache_reset(h)
    finally:
        K.kivi_cache_destroy(h)


def test_oracle_is_not_imported_by_the_library():
    pkg = os.path.join(ROOT, "bit_kivi_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"^\s*(?:from|import)\s+(\w+)", text, flags=re.M), f
