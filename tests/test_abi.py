"""The C ABI library loads, exports what include/nk.h declares, and rejects
host-checkable argument errors before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(nk_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_function():
    L = nk.lib()
    decl = declared_functions()
    assert decl, "no declarations found"
    missing = [n for n in sorted(decl) if not hasattr(L, n)]
    assert not missing, missing
    assert set(_lib.EXPORTS) == decl


def test_version_and_status_strings():
    assert nk.lib().nk_version() >= 100
    for code in range(8):
        s = nk.status_string(code)
        assert s and s != "unknown status"
    assert nk.status_string(99) == "unknown status"


@pytest.mark.parametrize("P,D,H,N", [(16, 64, 1, 16), (64, 256, 4, 512), (32, 128, 8, 3), (256, 256, 2, 7)])
def test_pool_size_agrees_with_the_oracle_layout(P, D, H, N):
    assert nk.kv_chunk_bytes(P, D) == oracle.chunk_bytes(P, D)
    assert nk.kv_pool_bytes(N, P, H, D) == oracle.pool_bytes(N, P, H, D)
    assert nk.kv_chunk_bytes(P, D) % 16 == 0


def test_chunk_bytes_rejects_bad_sizes():
    assert nk.kv_chunk_bytes(64, 100) == 0
    assert nk.kv_chunk_bytes(0, 256) == 0


def test_workspace_bytes_formula():
    # (num_ctas + B*Hkv) partial slots of T*G rows, D fp32 + 1 fp32 LSE each, 256-byte rounded
    n = nk.decode_workspace_bytes(8, 4, 24, 4, 256, 152)
    rows = (152 + 32) * 6 * 4
    assert n == ((rows * 257 * 4 + 255) // 256) * 256


FAKE = 1 << 20  # never dereferenced: every call below fails host validation first


def pool(num_pages=16, P=16, H=1, D=64, base=FAKE):
    return _lib.nk_kv_pool(base, num_pages, P, H, D)


def decode(p, T=1, Hq=2, B=1, max_ctx=64, max_pages=4, q=FAKE, out=FAKE, ws=FAKE, wsb=1 << 30, scale=0.125):
    L = nk.lib()
    return L.nk_paged_decode_attn(ctypes.byref(p) if p is not None else None, q, FAKE, max_pages, FAKE, B, T, Hq,
                                  scale, max_ctx, 0, ws, wsb, out, None, None)


def test_decode_rejects_bad_arguments():
    E = nk
    assert decode(None) == 1                                   # NULL pool
    assert decode(pool(base=0)) == 1                           # NULL base
    assert decode(pool(P=24)) == 2                             # page size not a multiple of 16
    assert decode(pool(D=96)) == 2                             # head_dim not 64/128/256
    assert decode(pool(), T=0) == 2
    assert decode(pool(), T=17) == 2                           # above NK_MAX_T
    assert decode(pool(H=2), Hq=3) == 2                        # Hq not a multiple of Hkv
    assert decode(pool(), max_ctx=65, max_pages=4) == 2        # max_ctx beyond the table
    assert decode(pool(), scale=float("nan")) == 2
    assert decode(pool(), q=FAKE + 2) == 2                     # misaligned Q
    assert decode(pool(), q=0) == 1
    assert decode(pool(), B=2000) == 3                         # beyond the batch limit
    assert decode(pool(), B=1025) == 3                         # one past it (1,024 sequences)
    assert decode(pool(P=256, D=256), max_pages=1) == 3        # a 256-key page of head_dim 256: no two-stage ring
    # a split giving one mma.sync CTA more than 262,144 keys of one kv-head
    # (T = 1 at G = 6: the mma.sync kernel; 4 CTAs over a 2^20-key sequence)
    L = nk.lib()
    big = pool(num_pages=1 << 14, P=64, H=4, D=256)
    assert L.nk_paged_decode_attn(ctypes.byref(big), FAKE, FAKE, 1 << 14, FAKE, 1, 1, 24, 0.0625, 1 << 20, 4,
                                  FAKE, 1 << 40, FAKE, None, None) == 3
    # the same split for a verify whose last column chunk runs on mma.sync
    # (T = 13 at G = 6: chunks of 4, 4, 4 and 1 columns)
    assert L.nk_paged_decode_attn(ctypes.byref(big), FAKE, FAKE, 1 << 14, FAKE, 1, 13, 24, 0.0625, 1 << 20, 4,
                                  FAKE, 1 << 40, FAKE, None, None) == 3
    assert decode(pool(), B=0) == 0                            # nothing to do
    assert E.lib().nk_paged_decode_attn_simt(ctypes.byref(pool()), FAKE, FAKE, 4, FAKE, 1, 1, 16, 0.1, 64, 0,
                                             FAKE, 1 << 30, FAKE, None, None) == 3  # G > 8 on CUDA cores


def test_append_rejects_bad_arguments():
    L = nk.lib()
    p = pool()
    assert L.nk_kv_append(None, FAKE, 4, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 1
    assert L.nk_kv_append(ctypes.byref(p), None, 4, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 1
    assert L.nk_kv_append(ctypes.byref(p), FAKE, 0, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 2
    assert L.nk_kv_append(ctypes.byref(p), FAKE, 4, FAKE, FAKE, 1, 1, FAKE + 8, FAKE, None, None) == 2
    assert L.nk_kv_append(ctypes.byref(p), FAKE, 4, FAKE, FAKE, 1, 0, FAKE, FAKE, None, None) == 0
    assert L.nk_kv_append(ctypes.byref(pool(num_pages=0)), FAKE, 4, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 2


def test_decode_step_checks_both_calls_before_launching():
    """nk_decode_step returns the first argument error of the append or the
    attention before launching anything (no GPU is touched here)."""
    L = nk.lib()
    p = pool()

    def step(pp=p, bt=FAKE, sp=FAKE, cu=FAKE, total=1, k=FAKE, v=FAKE, q=FAKE, ctx=FAKE, B=1, T=1, Hq=4,
             scale=0.1, max_ctx=64, max_pages=4):
        return L.nk_decode_step(ctypes.byref(pp) if pp is not None else None, bt, max_pages, sp, cu, total, k, v, q,
                                ctx, B, T, Hq, scale, max_ctx, 0, FAKE, 1 << 30, FAKE, None, None)

    assert step(pp=None) == 1                 # NULL pool
    assert step(sp=None) == 1                 # append: NULL start positions
    assert step(k=FAKE + 8) == 2              # append: misaligned K
    assert step(q=0) == 1                     # attention: NULL Q
    assert step(T=0) == 2                     # attention: T < 1
    assert step(scale=float("inf")) == 2      # attention: non-finite scale
    assert step(pp=pool(H=2), Hq=3) == 2      # attention: Hq not a multiple of Hkv
    assert step(B=0, total=0) == 0            # nothing to do


def test_combine_rejects_bad_arguments():
    L = nk.lib()
    assert L.nk_attn_combine(FAKE, FAKE, 2, 4, 96, FAKE, None) == 3
    assert L.nk_attn_combine(None, FAKE, 2, 4, 64, FAKE, None) == 1
    assert L.nk_attn_combine(FAKE, FAKE, -1, 4, 64, FAKE, None) == 2
    assert L.nk_attn_combine(FAKE, FAKE, 2, 0, 64, FAKE, None) == 0


@pytest.mark.parametrize("P,D,H,N", [(16, 64, 1, 16), (64, 256, 4, 512), (32, 128, 8, 3), (256, 256, 2, 7)])
def test_rk8v4_pool_size_agrees_with_the_oracle_layout(P, D, H, N):
    assert nk.rk8v4_chunk_bytes(P, D) == oracle.rk_chunk_bytes(P, D)
    assert nk.rk8v4_pool_bytes(N, P, H, D) == oracle.rk_pool_bytes(N, P, H, D)
    assert nk.rk8v4_chunk_bytes(P, D) % 16 == 0
    assert nk.rk8v4_chunk_bytes(64, 100) == 0 and nk.rk8v4_chunk_bytes(0, 256) == 0


def test_rk8v4_calls_reject_bad_arguments():
    L = nk.lib()
    p = pool()
    assert L.nk_rk8v4_append(None, FAKE, 4, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 1
    assert L.nk_rk8v4_append(ctypes.byref(p), FAKE, 0, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == 2
    assert L.nk_rk8v4_append(ctypes.byref(p), FAKE, 4, FAKE, FAKE, 1, 1, FAKE, FAKE + 8, None, None) == 2
    assert L.nk_rk8v4_append(ctypes.byref(p), FAKE, 4, FAKE, FAKE, 1, 0, FAKE, FAKE, None, None) == 0

    def dec(pp=p, T=1, Hq=2, B=1, max_ctx=64, q=FAKE, scale=0.125):
        return L.nk_rk8v4_decode_attn(ctypes.byref(pp) if pp is not None else None, q, FAKE, 4, FAKE, B, T, Hq,
                                      scale, max_ctx, 0, FAKE, 1 << 30, FAKE, None, None)

    assert dec(pp=None) == 1
    assert dec(pp=pool(P=24)) == 2
    assert dec(T=0) == 2 and dec(T=17) == 2
    assert dec(pp=pool(H=2), Hq=3) == 2
    assert dec(q=FAKE + 2) == 2
    assert dec(scale=float("nan")) == 2
    assert dec(Hq=16) == 3  # G > 8 on CUDA cores
    assert dec(B=0) == 0


def test_pool_format_is_checked_by_the_binding():
    """An INT8 pool is refused by the rk8v4 calls and the other way round
    (the C ABI cannot tell the formats apart: the Python pool carries it)."""
    import torch

    st = torch.zeros(16, dtype=torch.uint8)
    for fmt, other in (("int8", "rk8v4"), ("rk8v4", "int8")):
        p = nk.KVPool(st, 1, 16, 1, 64, fmt)
        p.need(fmt)
        with pytest.raises(ValueError):
            p.need(other)
    with pytest.raises(ValueError):
        nk.KVPool.empty(1, 16, 1, 64, device="cpu", fmt="fp8")


def test_noalloc_array_size_matches_the_header():
    src = open(os.path.join(ROOT, "include", "nk.h")).read()
    m = re.search(r"#define\s+NK_NOALLOC_MAX_WORKSPACE\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "NK_NOALLOC_MAX_WORKSPACE not found in nk.h"
    assert nk.NOALLOC_MAX_WORKSPACE == int(m.group(1)) << int(m.group(2))


def test_default_splits_is_exported_under_both_names():
    L = nk.lib()
    for args in [(1, 4, 32768, 64), (8, 4, 65536, 64), (1, 1, 256, 16), (3, 2, 17, 16)]:
        n = L.nk_decode_default_splits(*args)
        assert n == L.nk_decode_default_ctas(*args) == nk.decode_default_splits(*args)
        assert 1 <= n <= args[0] * args[1] * ((args[2] + args[3] - 1) // args[3])
    assert L.nk_decode_default_splits(0, 4, 100, 16) == 1


def test_host_step_layout():
    """nk_step_host_layout: six regions in order, each at a multiple of 256
    bytes and large enough for its tensor; bad shapes give 0."""
    B, total, T, Hq, Hkv, D = 3, 7, 4, 24, 4, 256
    nbytes, offs = nk.step_host_layout(B, total, T, Hq, Hkv, D)
    sizes = [total * Hkv * D * 2, total * Hkv * D * 2, B * T * Hq * D * 2, B * 4, (B + 1) * 4, B * 4]
    assert all(o % 256 == 0 for o in offs)
    for i in range(6):
        end = offs[i + 1] if i < 5 else nbytes
        assert end - offs[i] >= sizes[i]
        assert end - offs[i] < sizes[i] + 256
    with pytest.raises(ValueError):
        nk.step_host_layout(0, total, T, Hq, Hkv, D)


def test_prefill_rejects_bad_arguments():
    """nk_paged_prefill_attn's host checks, all before any launch."""
    L = nk.lib()
    p = pool(P=64, D=128, H=2)

    def pf(pp=p, q=FAKE, out=FAKE, B=1, T=32, Hq=4, max_pages=4, max_ctx=64, scale=0.125):
        return L.nk_paged_prefill_attn(ctypes.byref(pp) if pp is not None else None, q, FAKE, max_pages, FAKE, B, T,
                                       Hq, scale, max_ctx, out, None, None)

    assert pf(pp=None) == 1
    assert pf(q=None) == 1 and pf(out=None) == 1
    assert pf(T=0) == 2 and pf(B=-1) == 2
    assert pf(Hq=3) == 2                      # Hq not a multiple of Hkv
    assert pf(max_ctx=16) == 2                # max_ctx < T
    assert pf(max_pages=0) == 2 and pf(max_ctx=300) == 2
    assert pf(q=FAKE + 8) == 2                # misaligned Q
    assert pf(scale=float("inf")) == 2
    assert pf(pp=pool(P=64, D=96, H=2)) != 0  # head dim outside 64 / 128 / 256
    assert pf(B=0) == 0                       # nothing to do


def test_plain_c_program_compiles_and_links_against_the_library(tmp_path):
    # the header is plain C (C99, no C++): tests/abi_step.c, a decode loop that
    # includes only include/nk.h and the CUDA runtime header, builds with the
    # host C compiler and links against libnk.so with no unresolved symbol
    import shutil
    import subprocess

    from quantized_paged_kv_cache_gb300 import _build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    nk.lib()  # builds libnk.so when it is missing
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    exe = str(tmp_path / "abi_step")
    subprocess.run([cc, "-std=c99", "-D_POSIX_C_SOURCE=199309L", "-O1", "-Wall", "-Wextra", "-Werror", "-o", exe,
                    os.path.join(ROOT, "tests", "abi_step.c"), "-I", _build.INCLUDE,
                    "-I", os.path.join(cuda, "include"), "-L", os.path.dirname(_build.LIB), "-lnk",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,--no-undefined"], check=True)
    assert os.path.getsize(exe) > 0
