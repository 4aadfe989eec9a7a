"""fp64 CPU oracle for the paged INT8 group-64 KV cache -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package. The product path (``quantized_paged_kv_cache_gb300``) never does,
and the two share no code. The arithmetic lives in ``oracle.c`` (plain C,
fp64); this module only builds it with gcc and marshals numpy arrays through
ctypes.

Definitions and the readings of the NInfer README pages that they follow are
stated in ``oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (skipped when up to date)."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of every exported function."""
    P, I, D, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
    L.oracle_bf16_to_double.argtypes, L.oracle_bf16_to_double.restype = [ctypes.c_uint16], D
    L.oracle_double_to_bf16.argtypes, L.oracle_double_to_bf16.restype = [D], ctypes.c_uint16
    L.oracle_round_bf16.argtypes, L.oracle_round_bf16.restype = [P, Z, P], None
    L.oracle_quantize_group.argtypes, L.oracle_quantize_group.restype = [P, I, P], ctypes.c_float
    L.oracle_chunk_bytes.argtypes, L.oracle_chunk_bytes.restype = [I, I], Z
    L.oracle_pool_bytes.argtypes, L.oracle_pool_bytes.restype = [I, I, I, I], Z
    L.oracle_kv_append.argtypes = [P, I, I, I, I, P, I, P, P, I, P, P]
    L.oracle_kv_append.restype = I
    L.oracle_attention_row.argtypes = [P, I, I, I, I, P, I, P, I, I, I, P, D, I, I, I, I, I, P, P]
    L.oracle_attention_row.restype = I
    L.oracle_paged_attention.argtypes = [P, I, I, I, I, P, I, P, I, I, I, P, D, P, P]
    L.oracle_paged_attention.restype = I
    L.oracle_combine.argtypes, L.oracle_combine.restype = [P, P, I, I, I, P], None
    L.oracle_num_threads.argtypes, L.oracle_num_threads.restype = [], I
    U16 = ctypes.c_uint16
    L.oracle_double_to_f16.argtypes, L.oracle_double_to_f16.restype = [D], U16
    L.oracle_f16_to_double.argtypes, L.oracle_f16_to_double.restype = [U16], D
    L.oracle_rk_rotate64.argtypes, L.oracle_rk_rotate64.restype = [P, P], None
    L.oracle_rk_quantize_k.argtypes, L.oracle_rk_quantize_k.restype = [P, P], U16
    L.oracle_rk_quantize_v.argtypes, L.oracle_rk_quantize_v.restype = [P, P], U16
    L.oracle_rk_chunk_bytes.argtypes, L.oracle_rk_chunk_bytes.restype = [I, I], Z
    L.oracle_rk_pool_bytes.argtypes, L.oracle_rk_pool_bytes.restype = [I, I, I, I], Z
    L.oracle_rk_append.argtypes = [P, I, I, I, I, P, I, P, P, I, P, P]
    L.oracle_rk_append.restype = I
    L.oracle_rk_attention_row.argtypes = [P, I, I, I, I, P, I, P, I, I, I, P, D, I, I, I, I, I, P, P]
    L.oracle_rk_attention_row.restype = I
    L.oracle_rk_paged_attention.argtypes = [P, I, I, I, I, P, I, P, I, I, I, P, D, P, P]
    L.oracle_rk_paged_attention.restype = I
    L.oracle_i8h_quantize_group.argtypes, L.oracle_i8h_quantize_group.restype = [P, P], U16
    L.oracle_i8h_chunk_bytes.argtypes, L.oracle_i8h_chunk_bytes.restype = [I, I], Z
    L.oracle_bf16kv_chunk_bytes.argtypes, L.oracle_bf16kv_chunk_bytes.restype = [I, I], Z
    L.oracle_fmt_append.argtypes = [I, P, I, I, I, I, P, I, P, P, I, P, P]
    L.oracle_fmt_append.restype = I
    L.oracle_fmt_paged_attention.argtypes = [I, P, I, I, I, I, P, I, P, I, I, I, P, D, P, P]
    L.oracle_fmt_paged_attention.restype = I
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def use_library(path: str) -> None:
    """Make every wrapper below call the oracle compiled at `path` instead of
    liboracle.so (the tests use this to run the pins against deliberately
    altered copies of oracle.c)."""
    global _lib
    with _lock:
        _lib = _bind(ctypes.CDLL(os.path.abspath(path)))


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous, "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of raw bit patterns."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        import torch  # only for the view; no arithmetic

        return np.ascontiguousarray(x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    a = np.asarray(x)
    assert a.dtype == np.uint16, "bf16 input must be given as uint16 bit patterns or a torch.bfloat16 tensor"
    return np.ascontiguousarray(a)


def i32(x) -> np.ndarray:
    if hasattr(x, "cpu"):
        x = x.cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


# ---------------------------------------------------------------------------
# wrappers
# ---------------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def double_to_bf16(x: float) -> int:
    return lib().oracle_double_to_bf16(float(x))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (uint16), ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_round_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bits_to_double(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (data movement only)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def quantize_group(x_bits) -> tuple[np.ndarray, float]:
    x = _bits(x_bits).reshape(-1)
    q = np.empty(x.size, dtype=np.int8)
    s = lib().oracle_quantize_group(_ptr(x), x.size, _ptr(q))
    return q, float(np.float32(s))


def chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().oracle_chunk_bytes(page_size, head_dim))


def pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().oracle_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


def new_pool(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int, fill: int = 0) -> np.ndarray:
    return np.full(pool_bytes(num_pages, page_size, num_kv_heads, head_dim), fill, dtype=np.uint8)


def kv_append(pool: np.ndarray, num_pages, page_size, num_kv_heads, head_dim, block_table,
              start_pos, cu_new, k, v) -> int:
    bt = i32(block_table)
    sp, cu = i32(start_pos), i32(cu_new)
    kb, vb = _bits(k), _bits(v)
    assert pool.dtype == np.uint8 and pool.size >= pool_bytes(num_pages, page_size, num_kv_heads, head_dim)
    B = sp.size
    assert cu.size == B + 1 and kb.size == int(cu[-1]) * num_kv_heads * head_dim and vb.size == kb.size
    max_pages = bt.shape[1] if bt.ndim == 2 else bt.size // max(B, 1)
    return lib().oracle_kv_append(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                  max_pages, _ptr(sp), _ptr(cu), B, _ptr(kb), _ptr(vb))


def attention_row(pool, num_pages, page_size, num_kv_heads, head_dim, block_table, ctx_lens, q,
                  T, num_q_heads, sm_scale, b, t, i, key_begin=0, key_end=0x7FFFFFFF):
    bt, cl, qb = i32(block_table), i32(ctx_lens), _bits(q)
    B = cl.size
    o = np.empty(head_dim, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    rc = lib().oracle_attention_row(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                    bt.shape[1], _ptr(cl), B, T, num_q_heads, _ptr(qb), float(sm_scale),
                                    b, t, i, key_begin, key_end, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_attention_row: out-of-range data")
    return o, float(lse[0])


def paged_attention(pool, num_pages, page_size, num_kv_heads, head_dim, block_table, ctx_lens, q,
                    T, num_q_heads, sm_scale, want_lse=False):
    """fp64 output [B][T][Hq][D] (and lse [B][T][Hq])."""
    bt, cl, qb = i32(block_table), i32(ctx_lens), _bits(q)
    B = cl.size
    out = np.empty((B, T, num_q_heads, head_dim), dtype=np.float64)
    lse = np.empty((B, T, num_q_heads), dtype=np.float64)
    rc = lib().oracle_paged_attention(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                      bt.shape[1], _ptr(cl), B, T, num_q_heads, _ptr(qb), float(sm_scale),
                                      _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_paged_attention: {rc} rows with out-of-range data")
    return (out, lse) if want_lse else out


def combine(part_o: np.ndarray, part_lse: np.ndarray) -> np.ndarray:
    """part_o [S][R][D] fp32, part_lse [S][R] fp32 -> fp64 [R][D]."""
    po = np.ascontiguousarray(part_o, dtype=np.float32)
    pl = np.ascontiguousarray(part_lse, dtype=np.float32)
    S, R, D = po.shape
    assert pl.shape == (S, R)
    out = np.empty((R, D), dtype=np.float64)
    lib().oracle_combine(_ptr(po), _ptr(pl), S, R, D, _ptr(out))
    return out


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def chunk_view(pool: np.ndarray, num_pages, page_size, num_kv_heads, head_dim):
    """Split a pool byte array into (Kc, Ks, Vc, Vs) views of shape
    [pages][heads][P][D] / [pages][heads][P][D/64] (layout from oracle.h)."""
    P, D, g = page_size, head_dim, head_dim // 64
    cb = chunk_bytes(P, D)
    c = pool[: num_pages * num_kv_heads * cb].reshape(num_pages, num_kv_heads, cb)
    o1, o2, o3 = P * D, P * D + P * g * 4, 2 * P * D + P * g * 4
    kc = c[:, :, :o1].view(np.int8).reshape(num_pages, num_kv_heads, P, D)
    ks = c[:, :, o1:o2].copy().view(np.float32).reshape(num_pages, num_kv_heads, P, g)
    vc = c[:, :, o2:o3].view(np.int8).reshape(num_pages, num_kv_heads, P, D)
    vs = c[:, :, o3:].copy().view(np.float32).reshape(num_pages, num_kv_heads, P, g)
    return kc, ks, vc, vs


# ---------------------------------------------------------------------------
# rk8v4 (readings and layout in oracle.h)
# ---------------------------------------------------------------------------

def double_to_f16(x: float) -> int:
    return int(lib().oracle_double_to_f16(float(x)))


def f16_to_double(bits: int) -> float:
    return float(lib().oracle_f16_to_double(int(bits)))


def rk_rotate64(x_bits) -> np.ndarray:
    """R x of one 64-channel bf16 group: RN_fp32 of the exact H64 x / 8."""
    x = _bits(x_bits).reshape(-1)
    assert x.size == 64
    y = np.empty(64, dtype=np.float32)
    lib().oracle_rk_rotate64(_ptr(x), _ptr(y))
    return y


def rk_quantize_k(y) -> tuple[np.ndarray, int]:
    """64 rotated fp32 values -> (int8 codes, fp16 scale bits)."""
    y = np.ascontiguousarray(y, dtype=np.float32).reshape(-1)
    assert y.size == 64
    q = np.empty(64, dtype=np.int8)
    sb = lib().oracle_rk_quantize_k(_ptr(y), _ptr(q))
    return q, int(sb)


def rk_quantize_v(x_bits) -> tuple[np.ndarray, int]:
    """32 bf16 values -> (16 packed bytes, fp16 scale bits)."""
    x = _bits(x_bits).reshape(-1)
    assert x.size == 32
    packed = np.empty(16, dtype=np.uint8)
    sb = lib().oracle_rk_quantize_v(_ptr(x), _ptr(packed))
    return packed, int(sb)


def rk_chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().oracle_rk_chunk_bytes(page_size, head_dim))


def rk_pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().oracle_rk_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


def rk_new_pool(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int, fill: int = 0) -> np.ndarray:
    return np.full(rk_pool_bytes(num_pages, page_size, num_kv_heads, head_dim), fill, dtype=np.uint8)


def rk_append(pool: np.ndarray, num_pages, page_size, num_kv_heads, head_dim, block_table,
              start_pos, cu_new, k, v) -> int:
    bt = i32(block_table)
    sp, cu = i32(start_pos), i32(cu_new)
    kb, vb = _bits(k), _bits(v)
    assert pool.dtype == np.uint8 and pool.size >= rk_pool_bytes(num_pages, page_size, num_kv_heads, head_dim)
    B = sp.size
    assert cu.size == B + 1 and kb.size == int(cu[-1]) * num_kv_heads * head_dim and vb.size == kb.size
    max_pages = bt.shape[1] if bt.ndim == 2 else bt.size // max(B, 1)
    return lib().oracle_rk_append(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                  max_pages, _ptr(sp), _ptr(cu), B, _ptr(kb), _ptr(vb))


def rk_attention_row(pool, num_pages, page_size, num_kv_heads, head_dim, block_table, ctx_lens, q,
                     T, num_q_heads, sm_scale, b, t, i, key_begin=0, key_end=0x7FFFFFFF):
    bt, cl, qb = i32(block_table), i32(ctx_lens), _bits(q)
    o = np.empty(head_dim, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    rc = lib().oracle_rk_attention_row(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                       bt.shape[1], _ptr(cl), cl.size, T, num_q_heads, _ptr(qb), float(sm_scale),
                                       b, t, i, key_begin, key_end, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_rk_attention_row: out-of-range data")
    return o, float(lse[0])


def rk_paged_attention(pool, num_pages, page_size, num_kv_heads, head_dim, block_table, ctx_lens, q,
                       T, num_q_heads, sm_scale, want_lse=False):
    """fp64 output [B][T][Hq][D] (and lse [B][T][Hq]) over an rk8v4 pool."""
    bt, cl, qb = i32(block_table), i32(ctx_lens), _bits(q)
    B = cl.size
    out = np.empty((B, T, num_q_heads, head_dim), dtype=np.float64)
    lse = np.empty((B, T, num_q_heads), dtype=np.float64)
    rc = lib().oracle_rk_paged_attention(_ptr(pool), num_pages, page_size, num_kv_heads, head_dim, _ptr(bt),
                                         bt.shape[1], _ptr(cl), B, T, num_q_heads, _ptr(qb), float(sm_scale),
                                         _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_rk_paged_attention: {rc} rows with out-of-range data")
    return (out, lse) if want_lse else out


def rk_chunk_view(pool: np.ndarray, num_pages, page_size, num_kv_heads, head_dim):
    """Split an rk8v4 pool into (Kc int8 [pages][heads][P][D], Ks fp16 bits [..][P][D/64],
    Vc packed uint8 [..][P][D/2], Vs fp16 bits [..][P][D/32]) (layout from oracle.h)."""
    P, D = page_size, head_dim
    cb = rk_chunk_bytes(P, D)
    c = pool[: num_pages * num_kv_heads * cb].reshape(num_pages, num_kv_heads, cb)
    o1 = P * D
    o2 = o1 + P * (D // 64) * 2
    o3 = o2 + P * (D // 2)
    kc = c[:, :, :o1].view(np.int8).reshape(num_pages, num_kv_heads, P, D)
    ks = c[:, :, o1:o2].copy().view(np.uint16).reshape(num_pages, num_kv_heads, P, D // 64)
    vc = c[:, :, o2:o3].reshape(num_pages, num_kv_heads, P, D // 2)
    vs = c[:, :, o3:].copy().view(np.uint16).reshape(num_pages, num_kv_heads, P, D // 32)
    return kc, ks, vc, vs


# ---------------------------------------------------------------------------
# The pages' own INT8 layout (fp16 scales) and the bf16 baseline (oracle.h)
# ---------------------------------------------------------------------------
FORMATS = {"int8_f16": 1, "bf16": 2}


def i8h_quantize_group(x_bits) -> tuple[np.ndarray, int]:
    """64 bf16 values -> (int8 codes, fp16 scale bits)."""
    x = _bits(x_bits).reshape(-1)
    assert x.size == 64
    q = np.empty(64, dtype=np.int8)
    sb = lib().oracle_i8h_quantize_group(_ptr(x), _ptr(q))
    return q, int(sb)


def fmt_chunk_bytes(fmt: str, page_size: int, head_dim: int) -> int:
    f = lib().oracle_i8h_chunk_bytes if fmt == "int8_f16" else lib().oracle_bf16kv_chunk_bytes
    return int(f(page_size, head_dim))


def fmt_new_pool(fmt: str, num_pages, page_size, num_kv_heads, head_dim, fill: int = 0) -> np.ndarray:
    return np.full(num_pages * num_kv_heads * fmt_chunk_bytes(fmt, page_size, head_dim), fill, dtype=np.uint8)


def fmt_append(fmt: str, pool: np.ndarray, num_pages, page_size, num_kv_heads, head_dim, block_table,
               start_pos, cu_new, k, v) -> int:
    bt = i32(block_table)
    sp, cu = i32(start_pos), i32(cu_new)
    kb, vb = _bits(k), _bits(v)
    assert pool.dtype == np.uint8 and pool.size >= num_pages * num_kv_heads * fmt_chunk_bytes(fmt, page_size, head_dim)
    B = sp.size
    assert cu.size == B + 1 and kb.size == int(cu[-1]) * num_kv_heads * head_dim and vb.size == kb.size
    max_pages = bt.shape[1] if bt.ndim == 2 else bt.size // max(B, 1)
    return lib().oracle_fmt_append(FORMATS[fmt], _ptr(pool), num_pages, page_size, num_kv_heads, head_dim,
                                   _ptr(bt), max_pages, _ptr(sp), _ptr(cu), B, _ptr(kb), _ptr(vb))


def fmt_paged_attention(fmt: str, pool, num_pages, page_size, num_kv_heads, head_dim, block_table, ctx_lens, q,
                        T, num_q_heads, sm_scale, want_lse=False):
    bt, cl, qb = i32(block_table), i32(ctx_lens), _bits(q)
    B = cl.size
    out = np.empty((B, T, num_q_heads, head_dim), dtype=np.float64)
    lse = np.empty((B, T, num_q_heads), dtype=np.float64)
    rc = lib().oracle_fmt_paged_attention(FORMATS[fmt], _ptr(pool), num_pages, page_size, num_kv_heads, head_dim,
                                          _ptr(bt), bt.shape[1], _ptr(cl), B, T, num_q_heads, _ptr(qb),
                                          float(sm_scale), _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fmt_paged_attention: {rc} rows with out-of-range data")
    return (out, lse) if want_lse else out
