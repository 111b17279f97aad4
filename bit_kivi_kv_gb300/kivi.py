"""Python binding of the C ABI in include/kivi.h (ctypes; marshalling only).

The module-level functions carry the C names and take plain integers for
pointers and streams.  ``KiviCache`` wraps one handle with torch tensors for
device memory and the current torch stream.  Every computation runs in the
library's CUDA kernels; importing this module fails loudly when libkivi.so is
missing (build it with ``python -m bit_kivi_kv_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkivi.so")

KIVI_OK, KIVI_ERR_INVALID_ARG, KIVI_ERR_UNSUPPORTED, KIVI_ERR_CAPACITY, KIVI_ERR_STATE, KIVI_ERR_CUDA = range(6)
STATUS_NAMES = ["KIVI_OK", "KIVI_ERR_INVALID_ARG", "KIVI_ERR_UNSUPPORTED", "KIVI_ERR_CAPACITY",
                "KIVI_ERR_STATE", "KIVI_ERR_CUDA"]


class kivi_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("bits", ctypes.c_int), ("group", ctypes.c_int),
                ("residual", ctypes.c_int), ("max_tokens", ctypes.c_longlong)]


class kivi_layout(ctypes.Structure):
    _fields_ = [("total_bytes", ctypes.c_size_t), ("blocks_per_slot", ctypes.c_longlong),
                ("tile_bytes", ctypes.c_size_t), ("part_bytes", ctypes.c_size_t),
                ("slot_bytes", ctypes.c_size_t), ("k_resid_offset", ctypes.c_size_t),
                ("v_resid_offset", ctypes.c_size_t), ("resid_slot_bytes", ctypes.c_size_t)]


class kivi_paged_config(ctypes.Structure):
    _fields_ = [("max_seqs", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("bits", ctypes.c_int), ("group", ctypes.c_int),
                ("residual", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("n_pages", ctypes.c_longlong)]


class kivi_paged_layout(ctypes.Structure):
    _fields_ = [("total_bytes", ctypes.c_size_t), ("tile_bytes", ctypes.c_size_t),
                ("part_bytes", ctypes.c_size_t), ("page_bytes", ctypes.c_size_t),
                ("k_resid_offset", ctypes.c_size_t), ("v_resid_offset", ctypes.c_size_t),
                ("resid_seq_bytes", ctypes.c_size_t), ("table_offset", ctypes.c_size_t)]


KIVI_PAGED_MAX_CALL_SEQS = 512


class KiviError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 6 else status}: {message}")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m bit_kivi_kv_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, SZ, LL, I, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_longlong, ctypes.c_int, ctypes.c_float
    cfgp = ctypes.POINTER(kivi_config)
    pcfgp = ctypes.POINTER(kivi_paged_config)
    IP = ctypes.POINTER(ctypes.c_int)
    sigs = {
        "kivi_cache_bytes": (SZ, [cfgp]),
        "kivi_cache_layout": (I, [cfgp, ctypes.POINTER(kivi_layout)]),
        "kivi_cache_create": (I, [cfgp, P, SZ, ctypes.POINTER(P)]),
        "kivi_cache_destroy": (I, [P]),
        "kivi_cache_reset": (I, [P]),
        "kivi_cache_counts": (I, [P, ctypes.POINTER(LL), ctypes.POINTER(LL)]),
        "kivi_prefill": (I, [P, P, P, LL, P]),
        "kivi_append": (I, [P, P, P, P]),
        "kivi_decode_workspace_bytes": (SZ, [cfgp]),
        "kivi_decode_attn": (I, [P, P, P, F, P, SZ, P]),
        "kivi_append_decode": (I, [P, P, P, P, P, F, P, SZ, P]),
        "kivi_last_error_string": (ctypes.c_char_p, []),
        "kivi_launch_count": (ctypes.c_ulonglong, []),
        "kivi_cache_set_decode_kernel": (I, [P, I]),
        "kivi_cache_set_value_residual": (I, [P, I]),
        "kivi_cache_set_fault": (I, [P, I]),
        "kivi_cache_set_max_ctas": (I, [P, I]),
        "kivi_decode_attn_static_ws": (I, [P, P, P, F, P]),
        "kivi_paged_bytes": (SZ, [pcfgp]),
        "kivi_paged_cache_layout": (I, [pcfgp, ctypes.POINTER(kivi_paged_layout)]),
        "kivi_paged_create": (I, [pcfgp, P, SZ, ctypes.POINTER(P)]),
        "kivi_paged_destroy": (I, [P]),
        "kivi_paged_add": (I, [P, P, P, LL, P, IP]),
        "kivi_paged_release": (I, [P, I]),
        "kivi_paged_seq_counts": (I, [P, I, ctypes.POINTER(LL), ctypes.POINTER(LL)]),
        "kivi_paged_seq_pages": (I, [P, I, IP, I, IP]),
        "kivi_paged_free": (I, [P, ctypes.POINTER(LL), IP]),
        "kivi_paged_workspace_bytes": (SZ, [pcfgp, I]),
        "kivi_paged_set_max_ctas": (I, [P, I]),
        "kivi_paged_append_decode": (I, [P, IP, I, P, P, P, P, F, P, SZ, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


lib = _load()


def _check(status: int):
    if status != KIVI_OK:
        raise KiviError(status, lib.kivi_last_error_string().decode())


def make_config(batch, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_tokens) -> kivi_config:
    return kivi_config(batch, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_tokens)


# ---- the C calls, same names --------------------------------------------------
def kivi_cache_bytes(cfg: kivi_config) -> int:
    return lib.kivi_cache_bytes(ctypes.byref(cfg))


def kivi_cache_layout(cfg: kivi_config) -> kivi_layout:
    out = kivi_layout()
    _check(lib.kivi_cache_layout(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def kivi_cache_create(cfg: kivi_config, dev_buf: int, nbytes: int) -> int:
    h = ctypes.c_void_p()
    _check(lib.kivi_cache_create(ctypes.byref(cfg), dev_buf, nbytes, ctypes.byref(h)))
    return h.value


def kivi_cache_destroy(h: int):
    _check(lib.kivi_cache_destroy(h))


def kivi_cache_reset(h: int):
    _check(lib.kivi_cache_reset(h))


def kivi_cache_counts(h: int):
    a, b = ctypes.c_longlong(), ctypes.c_longlong()
    _check(lib.kivi_cache_counts(h, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def kivi_prefill(h: int, K: int, V: int, L: int, stream: int):
    _check(lib.kivi_prefill(h, K, V, L, stream))


def kivi_append(h: int, k: int, v: int, stream: int):
    _check(lib.kivi_append(h, k, v, stream))


def kivi_decode_workspace_bytes(cfg: kivi_config) -> int:
    return lib.kivi_decode_workspace_bytes(ctypes.byref(cfg))


def kivi_decode_attn(h: int, q: int, out: int, softmax_scale: float, workspace: int, ws_bytes: int, stream: int):
    _check(lib.kivi_decode_attn(h, q, out, softmax_scale, workspace, ws_bytes, stream))


def kivi_append_decode(h: int, k: int, v: int, q: int, out: int, softmax_scale: float, workspace: int,
                       ws_bytes: int, stream: int):
    _check(lib.kivi_append_decode(h, k, v, q, out, softmax_scale, workspace, ws_bytes, stream))


def kivi_decode_attn_static_ws(h: int, q: int, out: int, softmax_scale: float, stream: int):
    """Decode with the library's static workspace (for callers that cannot allocate)."""
    _check(lib.kivi_decode_attn_static_ws(h, q, out, softmax_scale, stream))


KIVI_DECODE_AUTO, KIVI_DECODE_CUDA_CORE, KIVI_DECODE_TENSOR_CORE = 0, 1, 2


def kivi_cache_set_decode_kernel(h: int, kernel: int):
    _check(lib.kivi_cache_set_decode_kernel(h, kernel))


KIVI_VALUE_FLUSH, KIVI_VALUE_QUEUE = 0, 1
KIVI_FAULT_NONE, KIVI_FAULT_COPY_STALL = 0, 1


def kivi_cache_set_max_ctas(h: int, max_ctas: int):
    _check(lib.kivi_cache_set_max_ctas(h, max_ctas))


def kivi_cache_set_fault(h: int, fault: int):
    """Failure-detection test hook (kivi.h): the next decode call's first copy stage in CTA 0 times out."""
    _check(lib.kivi_cache_set_fault(h, fault))


def kivi_cache_set_value_residual(h: int, mode: int):
    _check(lib.kivi_cache_set_value_residual(h, mode))


# ---- paged cache ----------------------------------------------------------------
def make_paged_config(max_seqs, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_blocks_per_seq,
                      n_pages) -> kivi_paged_config:
    return kivi_paged_config(max_seqs, n_q_heads, n_kv_heads, head_dim, bits, group, residual,
                             max_blocks_per_seq, n_pages)


def kivi_paged_bytes(cfg: kivi_paged_config) -> int:
    return lib.kivi_paged_bytes(ctypes.byref(cfg))


def kivi_paged_cache_layout(cfg: kivi_paged_config) -> kivi_paged_layout:
    out = kivi_paged_layout()
    _check(lib.kivi_paged_cache_layout(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def kivi_paged_create(cfg: kivi_paged_config, dev_buf: int, nbytes: int) -> int:
    h = ctypes.c_void_p()
    _check(lib.kivi_paged_create(ctypes.byref(cfg), dev_buf, nbytes, ctypes.byref(h)))
    return h.value


def kivi_paged_destroy(h: int):
    _check(lib.kivi_paged_destroy(h))


def kivi_paged_add(h: int, K: int, V: int, L: int, stream: int) -> int:
    s = ctypes.c_int()
    _check(lib.kivi_paged_add(h, K, V, L, stream, ctypes.byref(s)))
    return s.value


def kivi_paged_release(h: int, seq: int):
    _check(lib.kivi_paged_release(h, seq))


def kivi_paged_seq_counts(h: int, seq: int):
    a, b = ctypes.c_longlong(), ctypes.c_longlong()
    _check(lib.kivi_paged_seq_counts(h, seq, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def kivi_paged_seq_pages(h: int, seq: int) -> list:
    n = ctypes.c_int()
    _check(lib.kivi_paged_seq_pages(h, seq, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_int * max(n.value, 1))()
    _check(lib.kivi_paged_seq_pages(h, seq, buf, n.value, ctypes.byref(n)))
    return list(buf[:n.value])


def kivi_paged_free(h: int):
    a, b = ctypes.c_longlong(), ctypes.c_int()
    _check(lib.kivi_paged_free(h, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def kivi_paged_set_max_ctas(h: int, max_ctas: int):
    _check(lib.kivi_paged_set_max_ctas(h, max_ctas))


def kivi_paged_workspace_bytes(cfg: kivi_paged_config, n: int) -> int:
    return lib.kivi_paged_workspace_bytes(ctypes.byref(cfg), n)


def kivi_paged_append_decode(h: int, seqs, k: int, v: int, q: int, out: int, softmax_scale: float,
                             workspace: int, ws_bytes: int, stream: int):
    arr = (ctypes.c_int * max(len(seqs), 1))(*seqs)
    _check(lib.kivi_paged_append_decode(h, arr, len(seqs), k, v, q, out, softmax_scale, workspace, ws_bytes,
                                        stream))


def kivi_last_error_string() -> str:
    return lib.kivi_last_error_string().decode()


def kivi_launch_count() -> int:
    return lib.kivi_launch_count()


# ---- torch convenience wrapper -----------------------------------------------
class KiviCache:
    """One layer's cache: a torch-owned device buffer plus the library handle."""

    def __init__(self, batch, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_tokens,
                 device="cuda"):
        self.cfg = make_config(batch, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_tokens)
        nbytes = kivi_cache_bytes(self.cfg)
        if nbytes == 0:
            raise KiviError(KIVI_ERR_INVALID_ARG, kivi_last_error_string())
        self.layout = kivi_cache_layout(self.cfg)
        self.buffer = self._alloc(nbytes, device)
        self.workspace = self._alloc(kivi_decode_workspace_bytes(self.cfg), device)
        self.handle = kivi_cache_create(self.cfg, self.buffer.data_ptr(), nbytes)

    def _alloc(self, nbytes, device):
        """Device bytes for the cache buffer and the workspace (256-byte aligned);
        a subclass may place them differently (the tests put guard bands around them)."""
        import torch
        return torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.kivi_cache_destroy(h)
            self.handle = None

    @staticmethod
    def _stream(stream):
        import torch
        return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream

    @staticmethod
    def _ptr(t):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()

    def counts(self):
        return kivi_cache_counts(self.handle)

    def set_decode_kernel(self, kernel: int):
        kivi_cache_set_decode_kernel(self.handle, kernel)

    def set_value_residual(self, mode: int):
        """KIVI_VALUE_FLUSH (default) or KIVI_VALUE_QUEUE; on an empty cache."""
        kivi_cache_set_value_residual(self.handle, mode)

    def reset(self):
        kivi_cache_reset(self.handle)

    def prefill(self, K, V, stream=None):
        kivi_prefill(self.handle, self._ptr(K), self._ptr(V), K.shape[2], self._stream(stream))

    def append(self, k, v, stream=None):
        kivi_append(self.handle, self._ptr(k), self._ptr(v), self._stream(stream))

    def decode_attn(self, q, out=None, softmax_scale=0.0, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(q)
        kivi_decode_attn(self.handle, self._ptr(q), self._ptr(out), softmax_scale,
                         self.workspace.data_ptr(), self.workspace.numel(), self._stream(stream))
        return out

    def append_decode(self, k, v, q, out=None, softmax_scale=0.0, stream=None):
        """append(k, v) then decode_attn(q) in one call (one launch fewer)."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        kivi_append_decode(self.handle, self._ptr(k), self._ptr(v), self._ptr(q), self._ptr(out), softmax_scale,
                           self.workspace.data_ptr(), self.workspace.numel(), self._stream(stream))
        return out


class KiviPagedCache:
    """A paged cache for ragged sequences: a torch-owned device buffer (page pool,
    residual rows, block table) plus the library handle."""

    def __init__(self, max_seqs, n_q_heads, n_kv_heads, head_dim, bits, group, residual, max_blocks_per_seq,
                 n_pages, device="cuda"):
        self.cfg = make_paged_config(max_seqs, n_q_heads, n_kv_heads, head_dim, bits, group, residual,
                                     max_blocks_per_seq, n_pages)
        nbytes = kivi_paged_bytes(self.cfg)
        if nbytes == 0:
            raise KiviError(KIVI_ERR_INVALID_ARG, kivi_last_error_string())
        self.layout = kivi_paged_cache_layout(self.cfg)
        self.buffer = self._alloc(nbytes, device)
        self.workspace = self._alloc(kivi_paged_workspace_bytes(self.cfg, min(max_seqs, KIVI_PAGED_MAX_CALL_SEQS)),
                                     device)
        self.handle = kivi_paged_create(self.cfg, self.buffer.data_ptr(), nbytes)

    def _alloc(self, nbytes, device):
        """Device bytes for the buffer and the workspace (see KiviCache._alloc)."""
        import torch
        return torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.kivi_paged_destroy(h)
            self.handle = None

    def add(self, K, V, stream=None) -> int:
        """New sequence with prompt K, V [Hkv][L][D] fp16; returns its id."""
        L = K.shape[1]
        return kivi_paged_add(self.handle, KiviCache._ptr(K) if L else 0, KiviCache._ptr(V) if L else 0, L,
                              KiviCache._stream(stream))

    def release(self, seq: int):
        kivi_paged_release(self.handle, seq)

    def counts(self, seq: int):
        return kivi_paged_seq_counts(self.handle, seq)

    def pages(self, seq: int) -> list:
        return kivi_paged_seq_pages(self.handle, seq)

    def free(self):
        return kivi_paged_free(self.handle)

    def append_decode(self, seqs, k, v, q, out=None, softmax_scale=0.0, stream=None):
        """For each listed sequence: append k[i], v[i] ([n][Hkv][D]; both None: no
        append), then decode q[i] ([n][Hq][D]) into out[i]."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        kp = KiviCache._ptr(k) if k is not None else 0
        vp = KiviCache._ptr(v) if v is not None else 0
        kivi_paged_append_decode(self.handle, list(seqs), kp, vp, KiviCache._ptr(q), KiviCache._ptr(out),
                                 softmax_scale, self.workspace.data_ptr(), self.workspace.numel(),
                                 KiviCache._stream(stream))
        return out
