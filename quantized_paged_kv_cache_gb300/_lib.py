"""ctypes binding of ``libnk.so`` (argument marshalling only).

Every computation runs in the CUDA kernels behind the C ABI declared in
``include/nk.h``; this module only turns torch tensors into device pointers,
picks the current CUDA stream and raises on a nonzero status. There is no
CPU path: if the library cannot be loaded (or built), every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None


class NKError(RuntimeError):
    """A nonzero nk_status returned by the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: nk status {code} ({status_string(code)})")


class nk_kv_pool(ctypes.Structure):
    _fields_ = [
        ("base_dev", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
    ]


EXPORTS = (
    "nk_kv_chunk_bytes",
    "nk_kv_pool_bytes",
    "nk_kv_append",
    "nk_decode_default_splits",
    "nk_decode_default_ctas",
    "nk_decode_workspace_bytes",
    "nk_paged_decode_attn",
    "nk_paged_decode_attn_simt",
    "nk_paged_decode_attn_noalloc",
    "nk_decode_step",
    "nk_decode_step_host",
    "nk_step_host_layout",
    "nk_attn_combine",
    "nk_rk8v4_chunk_bytes",
    "nk_rk8v4_pool_bytes",
    "nk_rk8v4_append",
    "nk_rk8v4_decode_attn",
    "nk_i8f16_chunk_bytes",
    "nk_i8f16_pool_bytes",
    "nk_i8f16_append",
    "nk_i8f16_decode_attn",
    "nk_bf16kv_chunk_bytes",
    "nk_bf16kv_pool_bytes",
    "nk_bf16kv_append",
    "nk_bf16kv_decode_attn",
    "nk_status_string",
    "nk_version",
    "nk_test_inject_copy_stall",
    "nk_paged_prefill_attn",
)


def lib() -> ctypes.CDLL:
    """Load libnk.so, building it first when the sources are newer."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libnk.so is missing and could not be built")
            L = ctypes.CDLL(path)
            P, I32, Z, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
            pool_p = ctypes.POINTER(nk_kv_pool)
            L.nk_kv_chunk_bytes.argtypes, L.nk_kv_chunk_bytes.restype = [I32, I32], Z
            L.nk_kv_pool_bytes.argtypes, L.nk_kv_pool_bytes.restype = [I32, I32, I32, I32], Z
            L.nk_kv_append.argtypes = [pool_p, P, I32, P, P, I32, I32, P, P, P, P]
            L.nk_kv_append.restype = ctypes.c_int
            L.nk_decode_default_splits.argtypes, L.nk_decode_default_splits.restype = [I32, I32, I32, I32], I32
            L.nk_decode_default_ctas.argtypes, L.nk_decode_default_ctas.restype = [I32, I32, I32, I32], I32
            L.nk_decode_workspace_bytes.argtypes = [I32, I32, I32, I32, I32, I32]
            L.nk_decode_workspace_bytes.restype = Z
            dec = [pool_p, P, P, I32, P, I32, I32, I32, F, I32, I32, P, Z, P, P, P]
            L.nk_paged_decode_attn.argtypes, L.nk_paged_decode_attn.restype = dec, ctypes.c_int
            L.nk_paged_decode_attn_simt.argtypes, L.nk_paged_decode_attn_simt.restype = dec, ctypes.c_int
            L.nk_paged_decode_attn_noalloc.argtypes = [pool_p, P, P, I32, P, I32, I32, I32, F, I32, I32, P, P, P]
            L.nk_paged_decode_attn_noalloc.restype = ctypes.c_int
            L.nk_decode_step.argtypes = [pool_p, P, I32, P, P, I32, P, P, P, P, I32, I32, I32, F, I32, I32, P, Z, P,
                                         P, P]
            L.nk_decode_step.restype = ctypes.c_int
            L.nk_decode_step_host.argtypes = [pool_p, P, I32, I32, I32, I32, I32, F, I32, I32, P, P, P, Z, P, P, P,
                                              P, P]
            L.nk_decode_step_host.restype = ctypes.c_int
            L.nk_step_host_layout.argtypes = [I32, I32, I32, I32, I32, I32, ctypes.POINTER(ctypes.c_size_t)]
            L.nk_step_host_layout.restype = Z
            L.nk_rk8v4_chunk_bytes.argtypes, L.nk_rk8v4_chunk_bytes.restype = [I32, I32], Z
            L.nk_rk8v4_pool_bytes.argtypes, L.nk_rk8v4_pool_bytes.restype = [I32, I32, I32, I32], Z
            L.nk_rk8v4_append.argtypes = [pool_p, P, I32, P, P, I32, I32, P, P, P, P]
            L.nk_rk8v4_append.restype = ctypes.c_int
            L.nk_rk8v4_decode_attn.argtypes, L.nk_rk8v4_decode_attn.restype = dec, ctypes.c_int
            for fmt in ("i8f16", "bf16kv"):
                for name, args, res in ((f"nk_{fmt}_chunk_bytes", [I32, I32], Z),
                                        (f"nk_{fmt}_pool_bytes", [I32, I32, I32, I32], Z),
                                        (f"nk_{fmt}_append", [pool_p, P, I32, P, P, I32, I32, P, P, P, P], ctypes.c_int),
                                        (f"nk_{fmt}_decode_attn", dec, ctypes.c_int)):
                    fn = getattr(L, name)
                    fn.argtypes, fn.restype = args, res
            L.nk_paged_prefill_attn.argtypes = [pool_p, P, P, I32, P, I32, I32, I32, F, I32, P, P, P]
            L.nk_paged_prefill_attn.restype = ctypes.c_int
            L.nk_attn_combine.argtypes = [P, P, I32, I32, I32, P, P]
            L.nk_attn_combine.restype = ctypes.c_int
            L.nk_status_string.argtypes, L.nk_status_string.restype = [ctypes.c_int], ctypes.c_char_p
            L.nk_version.argtypes, L.nk_version.restype = [], ctypes.c_int
            L.nk_test_inject_copy_stall.argtypes = [I32, ctypes.c_uint64]
            L.nk_test_inject_copy_stall.restype = None
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().nk_status_string(int(code)).decode()
