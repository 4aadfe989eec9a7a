"""GPU parity of the pages' own INT8 layout (fp16 scales) and of the bf16 KV
baseline against the oracle ("NInfer-3090" README, "Choosing a KV format":
the int8 and bf16 rows of the table, 33,792 and 65,536 bytes per token).

The append must reproduce the oracle's pool bytes exactly (both formats);
i8f16 attention must meet the tolerance of the INT8 path against the
oracle's fp64 result, on the tcgen05 kernel (head_dim 256, 64-key pages,
9..32 rows per kv-head) and on the mma.sync kernel (every other shape). The
bf16 decode launches no kernel and must say so
(NK_ERR_UNSUPPORTED). Slots past the context hold 0xFF bytes (NaN scales or
values), which must not matter.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import Built, compare

pytestmark = pytest.mark.gpu

OFMT = {"i8f16": "int8_f16", "bf16": "bf16"}
APPEND = {"i8f16": nk.i8f16_append, "bf16": nk.bf16kv_append}
DECODE = {"i8f16": nk.i8f16_decode_attn, "bf16": nk.bf16kv_decode_attn}

CASES = {
    # name: (B, T, Hq, Hkv, D, P, ctx_lens)
    "d64_p16": (2, 1, 2, 1, 64, 16, [37, 300]),
    "d128_g3_t3": (3, 3, 6, 2, 128, 32, [3, 64, 517]),
    "d256_g6_t1": (2, 1, 24, 4, 256, 64, [130, 1900]),
    "d256_g6_t4": (3, 4, 24, 4, 256, 64, [4, 700, 2049]),    # i8f16: tcgen05
    "d256_g8_t2": (2, 2, 16, 2, 256, 16, [90, 333]),
    "d256_g6_t12": (2, 12, 24, 4, 256, 64, [12, 640]),       # column chunks
    "d64_g1_t16": (1, 16, 4, 4, 64, 16, [400]),
    "d256_p128_t3": (2, 3, 12, 2, 256, 128, [300, 1100]),
    "d256_g8_t6": (2, 6, 16, 2, 256, 32, [49, 900]),          # 48 rows: mma.sync, largest tile set
}


def build_fmt(fmt, w, fill=0x00, chunk=4096):
    c = Built()
    c.w = w
    c.bt_cpu = wl.block_table(w)
    c.bt = c.bt_cpu.cuda()
    c.ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    c.pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, fill=fill, fmt=fmt)
    c.opool = oracle.fmt_new_pool(OFMT[fmt], w.num_pages, w.P, w.Hkv, w.D, fill=fill)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(w.B):
        pos = 0
        while pos < w.ctx_lens[b]:
            n = min(chunk, w.ctx_lens[b] - pos)
            k, v = wl.kv_rows(w, b, pos, n)
            cu = torch.tensor([0, n], dtype=torch.int32)
            APPEND[fmt](c.pool, c.bt[b:b + 1].contiguous(), torch.tensor([pos], dtype=torch.int32, device="cuda"),
                        cu.cuda(), k.cuda(), v.cuda(), status=status)
            assert oracle.fmt_append(OFMT[fmt], c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu[b:b + 1], [pos],
                                     cu, k, v) == 0
            pos += n
    torch.cuda.synchronize()
    c.status = int(status.item())
    c.q = wl.queries(w).cuda()
    c.q_cpu = c.q.cpu()
    return c


def oracle_out(fmt, c):
    w = c.w
    return oracle.fmt_paged_attention(OFMT[fmt], c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu, w.ctx_lens,
                                      c.q_cpu, w.T, w.Hq, w.sm_scale)


def case(fmt, name, seed=8, fill=0xFF):
    B, T, Hq, Hkv, D, P, lens = CASES[name]
    w = wl.custom(f"{fmt}_{name}", B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=seed,
                  num_pages=sum((L + P - 1) // P for L in lens) + 3, outlier_channels=2, outlier_scale=8.0)
    return build_fmt(fmt, w, fill=fill)


@pytest.fixture(scope="module", params=[(f, n) for f in OFMT for n in CASES], ids=lambda x: f"{x[0]}-{x[1]}")
def built(request):
    fmt, name = request.param
    c = case(fmt, name)
    c.fmt = fmt
    c.ref = oracle_out(fmt, c)
    return c


def test_append_bit_exact(built):
    assert built.status == 0
    got = built.pool.storage.cpu().numpy()
    diff = np.flatnonzero(got != built.opool)
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"


def test_decode_matches_oracle(built):
    c, w = built, built.w
    if c.fmt == "bf16":
        # the library launches no kernel for a bf16 pool (see nk.h)
        with pytest.raises(nk.NKError) as ei:
            DECODE[c.fmt](c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
        assert ei.value.code == 3
        return
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = DECODE[c.fmt](c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, c.ref, f"{w.name}")
    again = DECODE[c.fmt](c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(out, again), "run-to-run results differ"
    for n in (1, 7, 300):
        o = DECODE[c.fmt](c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=n)
        torch.cuda.synchronize()
        compare(o, c.ref, f"{w.name}/ctas={n}")


@pytest.mark.parametrize("fmt", list(OFMT))
def test_append_ragged_batch_and_special_groups(fmt):
    """One call with unaligned starts, an empty sequence and page-crossing
    runs; groups of zeros, of tiny values (an fp16 scale below its range: 1,
    or subnormal), of huge values (fp16 saturation: the range flag)."""
    P, D, H = 16, 128, 2
    starts, lens = [5, 0, 31, 16], [40, 0, 3, 17]
    num_pages = 24
    rng = np.random.default_rng(9)
    bt = torch.from_numpy(rng.permutation(num_pages)[:4 * 6].reshape(4, 6).astype(np.int32))
    k = (torch.randn((sum(lens), H, D)) * 3).to(torch.bfloat16)
    v = torch.randn((sum(lens), H, D)).to(torch.bfloat16)
    k[0, 0, :64] = 0
    k[1, 0, :64] = torch.randn(64) * 2.0 ** -30     # a / 127 below the fp16 range
    k[2, 0, :64] = torch.randn(64) * 2.0 ** -18     # subnormal fp16 scale
    k[3, 1, 64:] = torch.randn(64) * 2.0 ** 30      # saturated scale
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int32)
    pool = nk.KVPool.empty(num_pages, P, H, D, fill=0x33, fmt=fmt)
    opool = oracle.fmt_new_pool(OFMT[fmt], num_pages, P, H, D, fill=0x33)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    APPEND[fmt](pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda(), status=status)
    assert oracle.fmt_append(OFMT[fmt], opool, num_pages, P, H, D, bt, sp, cu, k, v) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == (nk.NK_DEVFLAG_RANGE if fmt == "i8f16" else 0)
    assert np.array_equal(pool.storage.cpu().numpy(), opool)


@pytest.mark.parametrize("fmt", list(OFMT))
def test_streaming_append_bit_exact(fmt):
    """An append large enough for the streaming kernel (more than 4,096 groups),
    ragged over four sequences."""
    P, D, H = 64, 256, 4
    lens = [1000, 1, 777, 130]
    starts = [3, 64, 0, 500]
    num_pages = sum((s + n + P - 1) // P for s, n in zip(starts, lens)) + 2
    rng = np.random.default_rng(10)
    maxp = max((s + n + P - 1) // P for s, n in zip(starts, lens))
    perm = rng.permutation(num_pages)
    bt = np.full((4, maxp), -1, np.int32)
    off = 0
    for b in range(4):
        npg = (starts[b] + lens[b] + P - 1) // P
        bt[b, :npg] = perm[off:off + npg]
        off += npg
    bt = torch.from_numpy(bt)
    k = (torch.randn((sum(lens), H, D)) * torch.rand((sum(lens), H, 1)) * 4).to(torch.bfloat16)
    v = torch.randn((sum(lens), H, D)).to(torch.bfloat16)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int32)
    pool = nk.KVPool.empty(num_pages, P, H, D, fill=0x5A, fmt=fmt)
    opool = oracle.fmt_new_pool(OFMT[fmt], num_pages, P, H, D, fill=0x5A)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    APPEND[fmt](pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda(), status=status)
    assert oracle.fmt_append(OFMT[fmt], opool, num_pages, P, H, D, bt, sp, cu, k, v) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pool.storage.cpu().numpy(), opool)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["c1_i8f16"])
def test_full_size_c1(name):
    """The C1 decode workload (32,768 tokens) in each format, as bench.py runs
    it: the whole pool bit-exact, every output row within tolerance."""
    w = wl.make(name)
    c = build_fmt(w.fmt, w, fill=0, chunk=16384)
    assert c.status == 0
    assert np.array_equal(c.pool.storage.cpu().numpy(), c.opool)
    out = DECODE[w.fmt](c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    torch.cuda.synchronize()
    compare(out, oracle_out(w.fmt, c), name)
