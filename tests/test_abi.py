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


def test_paged_config_and_layout(K):
    cfg = K.make_paged_config(4, 32, 32, 128, 2, 32, 128, 16, 64)
    lay = K.kivi_paged_cache_layout(cfg)
    assert (lay.tile_bytes, lay.part_bytes) == (512, 1536)
    assert lay.page_bytes == 32 * 2 * 1536
    assert lay.k_resid_offset == 64 * lay.page_bytes                     # 256-aligned already
    assert lay.resid_seq_bytes == 32 * 128 * 128 * 2
    assert lay.v_resid_offset == lay.k_resid_offset + 4 * lay.resid_seq_bytes
    assert lay.table_offset == lay.v_resid_offset + 4 * lay.resid_seq_bytes
    assert lay.total_bytes == lay.table_offset + 4 * 16 * 4 == K.kivi_paged_bytes(cfg)
    assert K.kivi_paged_workspace_bytes(cfg, 3) == 3 * 32 * 65 * 132 * 4
    assert K.kivi_paged_workspace_bytes(cfg, 0) == 0
    assert K.kivi_paged_workspace_bytes(cfg, K.KIVI_PAGED_MAX_CALL_SEQS + 1) == 0
    bad = [K.make_paged_config(0, 32, 32, 128, 2, 32, 128, 16, 64),     # max_seqs
           K.make_paged_config(4, 32, 32, 128, 2, 32, 128, 0, 64),      # max_blocks_per_seq
           K.make_paged_config(4, 32, 32, 128, 2, 32, 128, 16, 0),      # n_pages
           K.make_paged_config(4, 32, 32, 128, 2, 32, 128, 16, 1 << 31),
           K.make_paged_config(4, 32, 32, 128, 3, 32, 128, 16, 64),     # bits
           K.make_paged_config(4, 32, 32, 128, 2, 32, 100, 16, 64)]     # residual % group
    for c in bad:
        assert K.kivi_paged_bytes(c) == 0
        assert K.kivi_last_error_string()


def test_paged_allocator_and_checks_without_gpu(K):
    """Sequence slots and pages come from host free lists; every check of
    add / append_decode runs before any launch, so failures leave the state as
    it was (fake device pointers are never dereferenced)."""
    cfg = K.make_paged_config(3, 2, 2, 64, 2, 32, 32, 4, 6)
    n = K.kivi_paged_bytes(cfg)
    fake = 1 << 20
    with pytest.raises(K.KiviError) as e:
        K.kivi_paged_create(cfg, fake + 16, n)
    assert e.value.status == K.KIVI_ERR_INVALID_ARG
    with pytest.raises(K.KiviError) as e:
        K.kivi_paged_create(cfg, fake, n - 1)
    assert e.value.status == K.KIVI_ERR_CAPACITY
    h = K.kivi_paged_create(cfg, fake, n)
    try:
        assert K.kivi_paged_free(h) == (6, 3)
        K.kivi_paged_set_max_ctas(h, 2)
        K.kivi_paged_set_max_ctas(h, 0)
        with pytest.raises(K.KiviError) as e:
            K.kivi_paged_set_max_ctas(h, -1)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        # empty prompts: no launch; slots handed out 0, 1, 2
        seqs = [K.kivi_paged_add(h, 0, 0, 0, 0) for _ in range(3)]
        assert seqs == [0, 1, 2] and K.kivi_paged_free(h) == (6, 0)
        assert K.kivi_paged_seq_counts(h, 1) == (0, 0) and K.kivi_paged_seq_pages(h, 1) == []
        with pytest.raises(K.KiviError) as e:          # no free slot
            K.kivi_paged_add(h, 0, 0, 0, 0)
        assert e.value.status == K.KIVI_ERR_CAPACITY
        K.kivi_paged_release(h, 1)
        assert K.kivi_paged_free(h) == (6, 1)
        with pytest.raises(K.KiviError) as e:          # released twice
            K.kivi_paged_release(h, 1)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        for bad in (-1, 3, 1):                          # out of range, out of range, not live
            with pytest.raises(K.KiviError) as e:
                K.kivi_paged_seq_counts(h, bad)
            assert e.value.status == K.KIVI_ERR_INVALID_ARG
        # a prompt of 4*32 + 32 + 1 tokens needs 5 blocks > max_blocks_per_seq 4
        with pytest.raises(K.KiviError) as e:
            K.kivi_paged_add(h, fake, fake, 161, 0)
        assert e.value.status == K.KIVI_ERR_CAPACITY
        with pytest.raises(K.KiviError) as e:          # misaligned prompt
            K.kivi_paged_add(h, fake + 8, fake, 10, 0)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        with pytest.raises(K.KiviError) as e:          # null prompt with L > 0
            K.kivi_paged_add(h, 0, 0, 10, 0)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        assert K.kivi_paged_free(h) == (6, 1)
        ws = K.kivi_paged_workspace_bytes(cfg, 2)
        ad = K.kivi_paged_append_decode
        cases = [(([0, 0], fake, fake, fake, fake, 0.0, fake, ws), K.KIVI_ERR_INVALID_ARG),   # listed twice
                 (([0, 1], fake, fake, fake, fake, 0.0, fake, ws), K.KIVI_ERR_INVALID_ARG),   # 1 is not live
                 (([], fake, fake, fake, fake, 0.0, fake, ws), K.KIVI_ERR_INVALID_ARG),       # n = 0
                 (([0, 2], fake, 0, fake, fake, 0.0, fake, ws), K.KIVI_ERR_INVALID_ARG),      # k without v
                 (([0, 2], fake + 8, fake + 8, fake, fake, 0.0, fake, ws), K.KIVI_ERR_INVALID_ARG),
                 (([0, 2], fake, fake, fake, fake, 0.0, fake + 64, ws), K.KIVI_ERR_INVALID_ARG),
                 (([0, 2], fake, fake, fake, fake, float("inf"), fake, ws), K.KIVI_ERR_INVALID_ARG),
                 (([0, 2], fake, fake, fake, fake, 0.0, fake, ws - 1), K.KIVI_ERR_CAPACITY),
                 (([0, 2], 0, 0, fake, fake, 0.0, fake, ws), K.KIVI_ERR_STATE)]           # decode only, empty
        for args, status in cases:
            with pytest.raises(K.KiviError) as e:
                ad(h, *args, 0)
            assert e.value.status == status, (args, e.value.status, K.kivi_last_error_string())
        with pytest.raises(K.KiviError) as e:          # more than KIVI_PAGED_MAX_CALL_SEQS sequences
            ad(h, [0] * (K.KIVI_PAGED_MAX_CALL_SEQS + 1), fake, fake, fake, fake, 0.0, fake, 1 << 40, 0)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        assert K.kivi_paged_free(h) == (6, 1)
        assert K.kivi_paged_seq_counts(h, 0) == (0, 0)
    finally:
        K.kivi_paged_destroy(h)


def test_value_residual_mode_checks_without_gpu(K):
    cfg = K.make_config(1, 2, 2, 64, 2, 32, 64, 256)
    fake = 1 << 20
    h = K.kivi_cache_create(cfg, fake, K.kivi_cache_bytes(cfg))
    try:
        K.kivi_cache_set_value_residual(h, K.KIVI_VALUE_QUEUE)
        K.kivi_cache_set_value_residual(h, K.KIVI_VALUE_FLUSH)
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_value_residual(h, 7)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
    finally:
        K.kivi_cache_destroy(h)
    big = K.make_config(1, 2, 2, 64, 2, 32, 256, 1024)     # residual > 128
    h = K.kivi_cache_create(big, fake, K.kivi_cache_bytes(big))
    try:
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_value_residual(h, K.KIVI_VALUE_QUEUE)
        assert e.value.status == K.KIVI_ERR_UNSUPPORTED
    finally:
        K.kivi_cache_destroy(h)


def test_fault_hook_argument_checks_without_gpu(K):
    cfg = K.make_config(1, 1, 1, 64, 2, 32, 32, 64)
    h = K.kivi_cache_create(cfg, 1 << 20, K.kivi_cache_bytes(cfg))
    try:
        K.kivi_cache_set_fault(h, K.KIVI_FAULT_COPY_STALL)
        K.kivi_cache_set_fault(h, K.KIVI_FAULT_NONE)
        K.kivi_cache_set_max_ctas(h, 3)
        K.kivi_cache_set_max_ctas(h, 0)
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_max_ctas(h, -1)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_fault(h, 5)
        assert e.value.status == K.KIVI_ERR_INVALID_ARG
    finally:
        K.kivi_cache_destroy(h)
