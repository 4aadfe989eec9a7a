"""Paged INT8 group-64 KV cache for one GB300: append, split-KV decode attention, combine.

The functions below mirror the C ABI in ``include/nk.h`` one to one and take
torch tensors that already live on the GPU. They only marshal arguments: the
work runs in the library's CUDA kernels on the current CUDA stream. Nothing
here synchronizes; errors in device data are reported through the optional
int32 ``status`` tensor (``NK_DEVFLAG_*`` bits).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from ._lib import NKError, lib, nk_kv_pool, status_string  # noqa: F401

NK_DEVFLAG_BAD_PAGE = 0x1
NK_DEVFLAG_BAD_POS = 0x2
NK_DEVFLAG_BAD_CTX = 0x4
NK_DEVFLAG_TIMEOUT = 0x8
NK_DEVFLAG_RANGE = 0x10
GROUP = 64
MAX_T = 16

__all__ = [
    "KVPool", "NKError", "kv_chunk_bytes", "kv_pool_bytes", "kv_append", "decode_default_splits", "decode_default_ctas",
    "decode_workspace_bytes", "paged_decode_attn", "paged_decode_attn_simt", "paged_decode_attn_noalloc",
    "attn_combine", "status_string", "decode_step", "rk8v4_chunk_bytes", "rk8v4_pool_bytes", "rk8v4_append",
    "rk8v4_decode_attn", "i8f16_chunk_bytes", "i8f16_pool_bytes", "i8f16_append", "i8f16_decode_attn",
    "bf16kv_chunk_bytes", "bf16kv_pool_bytes", "bf16kv_append", "bf16kv_decode_attn", "test_inject_copy_stall", "paged_prefill_attn",
]


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream))
    import torch

    return torch.cuda.current_stream().cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise NKError(rc, where)


def _need_cuda(*tensors) -> None:
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (there is no CPU path)")
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def kv_chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().nk_kv_chunk_bytes(page_size, head_dim))


def kv_pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().nk_kv_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


def i8f16_chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().nk_i8f16_chunk_bytes(page_size, head_dim))


def i8f16_pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().nk_i8f16_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


def bf16kv_chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().nk_bf16kv_chunk_bytes(page_size, head_dim))


def bf16kv_pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().nk_bf16kv_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


def rk8v4_chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(lib().nk_rk8v4_chunk_bytes(page_size, head_dim))


def rk8v4_pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().nk_rk8v4_pool_bytes(num_pages, page_size, num_kv_heads, head_dim))


@dataclass
class KVPool:
    """A caller-owned pool: ``storage`` is a uint8 CUDA tensor laid out as
    [page][kv-head][chunk], in the INT8 group-64 format with fp32 scales
    (``fmt="int8"``, ``kv_pool_bytes(...)`` bytes), the rk8v4 format
    (``"rk8v4"``), the pages' INT8 layout with fp16 scales (``"i8f16"``) or
    bf16 rows (``"bf16"``), each sized by its own ``*_pool_bytes``."""

    storage: "object"
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int
    fmt: str = "int8"

    @classmethod
    def empty(cls, num_pages, page_size, num_kv_heads, head_dim, device="cuda", fill: int | None = None,
              fmt: str = "int8"):
        import torch

        sizers = {"int8": kv_pool_bytes, "rk8v4": rk8v4_pool_bytes, "i8f16": i8f16_pool_bytes,
                  "bf16": bf16kv_pool_bytes}
        if fmt not in sizers:
            raise ValueError(f"unknown KV format {fmt!r}")
        n = sizers[fmt](num_pages, page_size, num_kv_heads, head_dim)
        st = torch.empty(n, dtype=torch.uint8, device=device)
        if fill is not None:
            st.fill_(fill)
        return cls(st, num_pages, page_size, num_kv_heads, head_dim, fmt)

    def need(self, fmt: str) -> None:
        if self.fmt != fmt:
            raise ValueError(f"this call needs a {fmt} pool, not a {self.fmt} one")

    def c_struct(self) -> nk_kv_pool:
        _need_cuda(self.storage)
        return nk_kv_pool(self.storage.data_ptr(), self.num_pages, self.page_size, self.num_kv_heads, self.head_dim)


def kv_append(pool: KVPool, block_table, start_pos, cu_new, k, v, status=None, stream=None) -> None:
    """Quantize k/v rows (bf16 [total_new][Hkv][D]) into the pool (nk_kv_append)."""
    _need_cuda(block_table, start_pos, cu_new, k, v, status)
    pool.need("int8")
    B = int(start_pos.numel())
    total = int(k.shape[0]) if k.dim() > 0 else 0
    ps = pool.c_struct()
    rc = lib().nk_kv_append(ctypes.byref(ps), _ptr(block_table), int(block_table.shape[-1]), _ptr(start_pos),
                            _ptr(cu_new), B, total, _ptr(k), _ptr(v), _ptr(status), _stream(stream))
    _check(rc, "nk_kv_append")


def decode_default_splits(B: int, num_kv_heads: int, max_ctx: int, page_size: int) -> int:
    """Default split (CTA) count of the decode calls (nk_decode_default_splits)."""
    return int(lib().nk_decode_default_splits(B, num_kv_heads, max_ctx, page_size))


def decode_default_ctas(B: int, num_kv_heads: int, max_ctx: int, page_size: int) -> int:
    """The same count under its earlier name (nk_decode_default_ctas)."""
    return int(lib().nk_decode_default_ctas(B, num_kv_heads, max_ctx, page_size))


def decode_workspace_bytes(B: int, T: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           num_ctas: int = 0) -> int:
    return int(lib().nk_decode_workspace_bytes(B, T, num_q_heads, num_kv_heads, head_dim, num_ctas))


def _decode(fn, name, pool, q, block_table, ctx_lens, sm_scale, max_ctx, num_ctas, workspace, out, status, stream,
            fmt="int8"):
    import torch

    _need_cuda(q, block_table, ctx_lens, workspace, out, status)
    pool.need(fmt)
    B, T, Hq, D = (int(s) for s in q.shape)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = decode_workspace_bytes(B, T, Hq, pool.num_kv_heads, D, num_ctas)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    ps = pool.c_struct()
    wbytes = workspace.numel() * workspace.element_size()
    rc = fn(ctypes.byref(ps), _ptr(q), _ptr(block_table), int(block_table.shape[-1]), _ptr(ctx_lens), B, T, Hq,
            float(sm_scale), int(max_ctx), int(num_ctas), _ptr(workspace), wbytes, _ptr(out), _ptr(status),
            _stream(stream))
    _check(rc, name)
    return out


def paged_decode_attn(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int, num_ctas: int = 0,
                      workspace=None, out=None, status=None, stream=None):
    """Split-KV paged attention on tensor cores (nk_paged_decode_attn); returns out bf16 [B][T][Hq][D]."""
    return _decode(lib().nk_paged_decode_attn, "nk_paged_decode_attn", pool, q, block_table, ctx_lens, sm_scale,
                   max_ctx, num_ctas, workspace, out, status, stream)


def paged_decode_attn_simt(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int,
                           num_ctas: int = 0, workspace=None, out=None, status=None, stream=None):
    """Same result from the fp32 CUDA-core kernel (nk_paged_decode_attn_simt)."""
    return _decode(lib().nk_paged_decode_attn_simt, "nk_paged_decode_attn_simt", pool, q, block_table, ctx_lens,
                   sm_scale, max_ctx, num_ctas, workspace, out, status, stream)


def decode_step(pool: KVPool, block_table, start_pos, cu_new, k, v, q, ctx_lens, sm_scale: float, max_ctx: int,
                num_ctas: int = 0, workspace=None, out=None, status=None, stream=None):
    """kv_append of the step's rows, then paged_decode_attn, in one call
    (nk_decode_step); returns out bf16 [B][T][Hq][D]."""
    import torch

    _need_cuda(block_table, start_pos, cu_new, k, v, q, ctx_lens, workspace, out, status)
    pool.need("int8")
    B, T, Hq, D = (int(s) for s in q.shape)
    if int(start_pos.numel()) != B:
        raise ValueError("start_pos must hold one position per sequence of q")
    total = int(k.shape[0]) if k.dim() > 0 else 0
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = decode_workspace_bytes(B, T, Hq, pool.num_kv_heads, D, num_ctas)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    ps = pool.c_struct()
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib().nk_decode_step(ctypes.byref(ps), _ptr(block_table), int(block_table.shape[-1]), _ptr(start_pos),
                              _ptr(cu_new), total, _ptr(k), _ptr(v), _ptr(q), _ptr(ctx_lens), B, T, Hq,
                              float(sm_scale), int(max_ctx), int(num_ctas), _ptr(workspace), wbytes, _ptr(out),
                              _ptr(status), _stream(stream))
    _check(rc, "nk_decode_step")
    return out


def step_host_layout(B: int, total_new: int, T: int, num_q_heads: int, num_kv_heads: int, head_dim: int):
    """(total bytes, offsets of k, v, q, start_pos, cu_new, ctx_lens) of
    decode_step_host's input buffer (nk_step_host_layout)."""
    offs = (ctypes.c_size_t * 6)()
    total = lib().nk_step_host_layout(int(B), int(total_new), int(T), int(num_q_heads), int(num_kv_heads),
                                      int(head_dim), offs)
    if total == 0:
        raise ValueError("invalid shape for the host step layout")
    return int(total), tuple(int(o) for o in offs)


def decode_step_host(pool: KVPool, block_table, B: int, total_new: int, T: int, num_q_heads: int, sm_scale: float,
                     max_ctx: int, in_host, staging, out, out_host, num_ctas: int = 0, workspace=None, status=None,
                     status_host=None, stream=None):
    """nk_decode_step_host: one step from host memory. in_host is a host
    uint8 tensor (pinned for an asynchronous transfer) in the
    step_host_layout layout; staging a device buffer of at least that size;
    out the device output [B][T][Hq][D] bf16 and out_host its host copy;
    status_host an int32 host tensor of one element. Waits for the stream."""
    import torch

    _need_cuda(block_table, staging, out, workspace, status)
    pool.need("int8")
    if in_host.is_cuda or out_host.is_cuda or (status_host is not None and status_host.is_cuda):
        raise ValueError("in_host, out_host and status_host must be host tensors")
    D = pool.head_dim
    if workspace is None:
        nbytes = decode_workspace_bytes(B, T, num_q_heads, pool.num_kv_heads, D, num_ctas)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=staging.device)
    ps = pool.c_struct()
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib().nk_decode_step_host(ctypes.byref(ps), _ptr(block_table), int(block_table.shape[-1]), int(B),
                                   int(total_new), int(T), int(num_q_heads), float(sm_scale), int(max_ctx),
                                   int(num_ctas), _ptr(in_host), _ptr(staging), _ptr(workspace), wbytes, _ptr(out),
                                   _ptr(out_host), _ptr(status), _ptr(status_host), _stream(stream))
    _check(rc, "nk_decode_step_host")
    return out_host


NOALLOC_MAX_WORKSPACE = 8 << 20


def paged_decode_attn_noalloc(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int,
                              num_ctas: int = 0, out=None, status=None, stream=None):
    """nk_paged_decode_attn_noalloc: the tensor-core decode with its split
    partials in the library's own fixed device array, for callers that cannot
    allocate device memory. Calls that overlap on the GPU race on that array."""
    import torch

    _need_cuda(q, block_table, ctx_lens, out, status)
    pool.need("int8")
    B, T, Hq, D = (int(s) for s in q.shape)
    if out is None:
        out = torch.empty_like(q)
    ps = pool.c_struct()
    rc = lib().nk_paged_decode_attn_noalloc(ctypes.byref(ps), _ptr(q), _ptr(block_table), int(block_table.shape[-1]),
                                            _ptr(ctx_lens), B, T, Hq, float(sm_scale), int(max_ctx), int(num_ctas),
                                            _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "nk_paged_decode_attn_noalloc")
    return out


def rk8v4_append(pool: KVPool, block_table, start_pos, cu_new, k, v, status=None, stream=None) -> None:
    """Rotate, quantize and scatter k/v rows (bf16 [total_new][Hkv][D]) into an rk8v4 pool (nk_rk8v4_append)."""
    _need_cuda(block_table, start_pos, cu_new, k, v, status)
    pool.need("rk8v4")
    B = int(start_pos.numel())
    total = int(k.shape[0]) if k.dim() > 0 else 0
    ps = pool.c_struct()
    rc = lib().nk_rk8v4_append(ctypes.byref(ps), _ptr(block_table), int(block_table.shape[-1]), _ptr(start_pos),
                               _ptr(cu_new), B, total, _ptr(k), _ptr(v), _ptr(status), _stream(stream))
    _check(rc, "nk_rk8v4_append")


def rk8v4_decode_attn(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int, num_ctas: int = 0,
                      workspace=None, out=None, status=None, stream=None):
    """Split-KV paged attention over an rk8v4 pool (nk_rk8v4_decode_attn); returns out bf16 [B][T][Hq][D]."""
    return _decode(lib().nk_rk8v4_decode_attn, "nk_rk8v4_decode_attn", pool, q, block_table, ctx_lens, sm_scale,
                   max_ctx, num_ctas, workspace, out, status, stream, fmt="rk8v4")


def attn_combine(part_o, part_lse, out=None, stream=None):
    """LSE merge of partials: part_o fp32 [S][R][D], part_lse fp32 [S][R] -> bf16 [R][D] (nk_attn_combine)."""
    import torch

    _need_cuda(part_o, part_lse, out)
    S, R, D = (int(s) for s in part_o.shape)
    if out is None:
        out = torch.empty((R, D), dtype=torch.bfloat16, device=part_o.device)
    rc = lib().nk_attn_combine(_ptr(part_o), _ptr(part_lse), S, R, D, _ptr(out), _stream(stream))
    _check(rc, "nk_attn_combine")
    return out


def test_inject_copy_stall(withheld_page: int, wait_cycles: int = 0) -> None:
    """nk_test_inject_copy_stall: failure injection for the bounded-wait tests
    (withheld_page < 0 switches it off)."""
    lib().nk_test_inject_copy_stall(int(withheld_page), int(wait_cycles))


def _fmt_append(fn, name, fmt, pool, block_table, start_pos, cu_new, k, v, status, stream):
    _need_cuda(block_table, start_pos, cu_new, k, v, status)
    pool.need(fmt)
    B = int(start_pos.numel())
    total = int(k.shape[0]) if k.dim() > 0 else 0
    ps = pool.c_struct()
    rc = fn(ctypes.byref(ps), _ptr(block_table), int(block_table.shape[-1]), _ptr(start_pos), _ptr(cu_new), B, total,
            _ptr(k), _ptr(v), _ptr(status), _stream(stream))
    _check(rc, name)


def i8f16_append(pool: KVPool, block_table, start_pos, cu_new, k, v, status=None, stream=None) -> None:
    """Quantize k/v rows into a pool of the pages' INT8 layout with fp16 scales (nk_i8f16_append)."""
    _fmt_append(lib().nk_i8f16_append, "nk_i8f16_append", "i8f16", pool, block_table, start_pos, cu_new, k, v,
                status, stream)


def bf16kv_append(pool: KVPool, block_table, start_pos, cu_new, k, v, status=None, stream=None) -> None:
    """Scatter bf16 k/v rows into a bf16 pool (nk_bf16kv_append)."""
    _fmt_append(lib().nk_bf16kv_append, "nk_bf16kv_append", "bf16", pool, block_table, start_pos, cu_new, k, v,
                status, stream)


def i8f16_decode_attn(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int, num_ctas: int = 0,
                      workspace=None, out=None, status=None, stream=None):
    """Split-KV paged attention over an INT8 pool with fp16 scales (nk_i8f16_decode_attn)."""
    return _decode(lib().nk_i8f16_decode_attn, "nk_i8f16_decode_attn", pool, q, block_table, ctx_lens, sm_scale,
                   max_ctx, num_ctas, workspace, out, status, stream, fmt="i8f16")


def bf16kv_decode_attn(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int, num_ctas: int = 0,
                       workspace=None, out=None, status=None, stream=None):
    """Split-KV paged attention over a bf16 pool (nk_bf16kv_decode_attn)."""
    return _decode(lib().nk_bf16kv_decode_attn, "nk_bf16kv_decode_attn", pool, q, block_table, ctx_lens, sm_scale,
                   max_ctx, num_ctas, workspace, out, status, stream, fmt="bf16")


def paged_prefill_attn(pool: KVPool, q, block_table, ctx_lens, sm_scale: float, max_ctx: int, out=None, status=None,
                       stream=None):
    """Chunked-prefill attention of T query tokens per sequence over the paged
    INT8 cache (nk_paged_prefill_attn); returns out bf16 [B][T][Hq][D]."""
    import torch

    _need_cuda(q, block_table, ctx_lens, out, status)
    pool.need("int8")
    B, T, Hq, D = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    ps = pool.c_struct()
    rc = lib().nk_paged_prefill_attn(ctypes.byref(ps), _ptr(q), _ptr(block_table), int(block_table.shape[-1]),
                                     _ptr(ctx_lens), B, T, Hq, float(sm_scale), int(max_ctx), _ptr(out), _ptr(status),
                                     _stream(stream))
    _check(rc, "nk_paged_prefill_attn")
    return out
