"""GPU parity: the CUDA kernels against the fp64 oracle on the same seeded inputs.

Append: int8 codes and fp32 scales bit-exact, over the whole pool.
Attention: max-abs <= 4e-3 and relative L2 <= 1e-3 against the oracle's fp64
output rounded to bf16, for the tensor-core kernel and the CUDA-core kernel.
Shapes span several pages and CTAs with ragged tails (unaligned context
lengths and append starts), T = 1..8 causal verify columns, GQA ratios and
page sizes; plus the degenerate cases (ctx = T, one key, empty sequences).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import ABS_TOL, REL_L2_TOL, build, compare, gpu_pool_bytes, oracle_attention_full, run_decode

pytestmark = pytest.mark.gpu
IMPLS = ["mma", "simt"]


def small(name, B, T, Hq, Hkv, D, P, lens, seed, num_pages=None, **kw):
    return wl.custom(name, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=seed, num_pages=num_pages, **kw)


SHAPES = [
    # name,           B, T, Hq, Hkv,  D,   P, lens
    ("tiny",          1, 1, 2, 1, 64, 16, [256]),
    ("t1_d256",       1, 1, 24, 4, 256, 64, [1000]),
    ("t4_d256",       2, 4, 24, 4, 256, 64, [700, 4099]),
    ("t2_d128",       3, 2, 16, 2, 128, 32, [33, 2, 515]),
    ("t8_d64",        2, 8, 8, 1, 64, 16, [8, 300]),       # M = 64: mma.sync in chunks of 6 columns
    ("t8_g6",         2, 8, 12, 2, 128, 16, [9, 700]),     # M = 48: largest tensor-core tile set
    ("t3_g8",         2, 3, 32, 4, 128, 16, [77, 1234]),
    ("t5_mix",        4, 5, 12, 4, 256, 16, [5, 64, 65, 3000]),
    ("t1_b8",         8, 1, 24, 4, 256, 64, [64, 1, 128, 129, 4000, 63, 1000, 2]),
    ("t4_p128",       2, 4, 24, 4, 256, 128, [255, 1025]),
    # the tcgen05 kernel's instances (D = 256, P = 64, 9 <= G*T <= 32)
    ("t2_tc",         3, 2, 24, 4, 256, 64, [100, 2, 700]),     # M = 12: two 8-row tiles
    ("t3_tc",         2, 3, 24, 4, 256, 64, [3, 1500]),         # M = 18: three tiles, rows padded to 32
    ("t4_g8_tc",      2, 4, 32, 4, 256, 64, [65, 900]),         # M = 32: four tiles
    ("t5_g2_tc",      5, 5, 8, 4, 256, 64, [5, 64, 65, 128, 2000]),  # M = 10, many short units
    # wide verifies: column chunks of 4 (tcgen05, 24 rows) or of 48 // G
    # columns (mma.sync); 8 on CUDA cores
    ("t8_chunks",     2, 8, 24, 4, 256, 64, [300, 2500]),     # M = 48: two chunks of 4
    ("t12_chunks",    2, 12, 24, 4, 256, 64, [12, 1500]),     # ctx = T; three chunks
    ("t16_g2_tc",     3, 16, 8, 4, 256, 64, [16, 700, 2000]), # M = 32: one tcgen05 launch
    ("t16_d128",      2, 16, 16, 2, 128, 32, [40, 900]),      # G = 8, M = 128: chunks of 6
    ("t16_p128",      1, 16, 24, 4, 256, 128, [3000]),        # mma.sync, 128-key pages: the largest chunk that fits
    ("t16_g1_tc",     2, 16, 4, 4, 256, 64, [20, 900]),       # G = 1: 16 rows, one tcgen05 launch
]


@pytest.fixture(scope="module", params=SHAPES, ids=[s[0] for s in SHAPES])
def case(request):
    name, B, T, Hq, Hkv, D, P, lens = request.param
    w = small(name, B, T, Hq, Hkv, D, P, lens, seed=zlib.crc32(name.encode()) % 1000, num_pages=sum((L + P - 1) // P for L in lens) + 5)
    c = build(w, fill=0)
    c.ref = oracle_attention_full(c)
    return c


def test_append_bit_exact(case):
    assert np.array_equal(gpu_pool_bytes(case), case.opool)


def unsupported(w, impl):
    """The tensor-core kernels hold at most 48 query rows per kv-head in one
    launch, so a column chunk needs G <= 48; the CUDA-core kernel G <= 8."""
    return (impl == "mma" and w.G > 48) or (impl == "simt" and w.G > 8)


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_matches_oracle(case, impl):
    if unsupported(case.w, impl):
        with pytest.raises(nk.NKError) as ei:
            run_decode(case, impl)
        assert ei.value.code == 3
        return
    out = run_decode(case, impl)
    torch.cuda.synchronize()
    compare(out, case.ref, f"{case.w.name}/{impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_is_deterministic_and_cta_count_independent(case, impl):
    if unsupported(case.w, impl):
        pytest.skip("shape outside the tensor-core kernel (checked in test_decode_matches_oracle)")
    a = run_decode(case, impl)
    b = run_decode(case, impl)
    torch.cuda.synchronize()
    assert torch.equal(a, b), "run-to-run results differ"
    for n in (1, 3, 7, 200):
        o = run_decode(case, impl, num_ctas=n)
        torch.cuda.synchronize()
        compare(o, case.ref, f"{case.w.name}/{impl}/ctas={n}")


@pytest.mark.parametrize("shape", [
    ("b1024_mma", 1, 8, 2, 128, 16),   # mma.sync kernel
    ("b1024_tc", 4, 24, 4, 256, 64),   # tcgen05 kernel (24 rows per kv-head)
], ids=lambda s: s[0])
def test_decode_at_the_batch_limit(shape):
    """1,024 sequences, the most one call takes (their page prefix sums live
    in shared memory), with short ragged contexts down to T keys, against the
    oracle on both tensor-core paths and the CUDA-core kernel."""
    name, T, Hq, Hkv, D, P = shape
    rng = np.random.default_rng(1024 + T)
    lens = [int(x) for x in rng.integers(T, 100, 1024)]
    lens[0], lens[-1] = T, 2 * P + 3
    w = small(name, 1024, T, Hq, Hkv, D, P, lens, seed=11, num_pages=sum((L + P - 1) // P for L in lens) + 4)
    c = build(w, fill=0)
    ref = oracle_attention_full(c)
    for impl in IMPLS:
        out = run_decode(c, impl)
        torch.cuda.synchronize()
        compare(out, ref, f"{name}/{impl}")


def test_append_ragged_starts_and_empty_sequences():
    """Several sequences, unaligned starts, one sequence with no new rows."""
    w = small("ragged", 4, 1, 8, 2, 128, 16, [50, 37, 90, 17], seed=5, num_pages=20)
    bt = wl.block_table(w).cuda()
    pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, fill=0)
    opool = oracle.new_pool(w.num_pages, w.P, w.Hkv, w.D)
    starts = [3, 0, 17, 16]
    lens = [40, 0, 73, 1]
    k, v, sp, cu = wl.append_batch(w, starts, lens, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.kv_append(pool, bt, sp.cuda(), cu.cuda(), k, v, status=status)
    torch.cuda.synchronize()
    assert oracle.kv_append(opool, w.num_pages, w.P, w.Hkv, w.D, wl.block_table(w), sp, cu, k.cpu(), v.cpu()) == 0
    assert int(status.item()) == 0
    assert np.array_equal(pool.storage.cpu().numpy(), opool)


@pytest.mark.parametrize("nseq", [5, 300])
def test_append_streaming_many_sequences(nseq):
    """The streaming kernel (more than 4,096 groups) over several sequences
    with unaligned starts and one empty sequence: up to 256 sequences its
    destination search reads cu_new from shared memory, beyond that from
    global memory."""
    rng = np.random.default_rng(nseq)
    lens = [int(x) for x in rng.integers(20, 200, nseq)]
    lens[1] = 0
    starts = [int(x) for x in rng.integers(0, 100, nseq)]
    P, D, Hkv = 16, 256, 4
    ctx = [s + n + 1 for s, n in zip(starts, lens)]
    w = small("stream_many", nseq, 1, 8, Hkv, D, P, ctx, seed=nseq, num_pages=sum((L + P - 1) // P for L in ctx) + 3)
    assert sum(lens) * Hkv * 2 * (D // 64) > 4096
    bt = wl.block_table(w).cuda()
    pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, fill=0)
    opool = oracle.new_pool(w.num_pages, w.P, w.Hkv, w.D)
    k, v, sp, cu = wl.append_batch(w, starts, lens, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.kv_append(pool, bt, sp.cuda(), cu.cuda(), k, v, status=status)
    torch.cuda.synchronize()
    assert oracle.kv_append(opool, w.num_pages, w.P, w.Hkv, w.D, wl.block_table(w), sp, cu, k.cpu(), v.cpu()) == 0
    assert int(status.item()) == 0
    assert np.array_equal(pool.storage.cpu().numpy(), opool)


def _bits_to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("copies", [1, 3])
def test_append_special_values(copies):
    """Exact ties, zero groups, negative zeros, huge and tiny magnitudes, and
    every finite bf16 bit pattern, quantized bit-exactly. One copy (about
    2,000 groups) takes the small-append kernel, three copies the streaming
    kernel."""
    D, H, P = 256, 2, 16
    rng = np.random.default_rng(3)
    rows = []
    # exact ties: absmax 15.875 -> s = 0.125, values k*0.125 + 0.0625
    g = np.zeros(64, np.float32)
    g[0] = 15.875
    g[1:40] = (np.arange(-19, 20) * 0.125 + 0.0625).astype(np.float32)
    rows.append(g)
    rows.append(np.zeros(64, np.float32))                    # a = 0
    rows.append(-np.zeros(64, np.float32))                   # negative zeros
    rows.append((rng.standard_normal(64) * 1e30).astype(np.float32))
    rows.append((rng.standard_normal(64) * 1e-35).astype(np.float32))
    rows.append(np.full(64, 3.0, np.float32))                # all equal
    groups = [torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for r in rows]
    # every finite bf16 pattern, in groups of 64 (absmax varies per group)
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    fin = allb[np.isfinite(oracle.bits_to_double(allb))]
    fin = fin[rng.permutation(fin.size)]
    pad = (-fin.size) % 64
    fin = np.concatenate([fin, np.zeros(pad, np.uint16)])
    groups += list(fin.reshape(-1, 64))
    groups = groups * copies
    n_groups = len(groups)
    per_row = H * D // 64
    n_rows = (n_groups + per_row - 1) // per_row
    flat = np.concatenate(groups + [np.zeros(64, np.uint16)] * (n_rows * per_row - n_groups))
    k = _bits_to_bf16(flat).reshape(n_rows, H, D)
    v = _bits_to_bf16(np.roll(flat, 64)).reshape(n_rows, H, D)
    pages = (n_rows + P - 1) // P
    bt = torch.arange(pages, dtype=torch.int32).flip(0)[None].contiguous()
    pool = nk.KVPool.empty(pages, P, H, D, fill=0xAB)
    opool = oracle.new_pool(pages, P, H, D, fill=0xAB)
    cu = torch.tensor([0, n_rows], dtype=torch.int32)
    sp = torch.tensor([0], dtype=torch.int32)
    nk.kv_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert oracle.kv_append(opool, pages, P, H, D, bt, sp, cu, k, v) == 0
    got = pool.storage.cpu().numpy()
    assert np.array_equal(got, opool)


def test_append_flags_bad_pages_and_positions():
    w = small("badpg", 1, 1, 2, 1, 64, 16, [40], seed=1, num_pages=4)
    bt = wl.block_table(w).clone()
    bt[0, 1] = 99                           # page outside the pool
    pool = nk.KVPool.empty(w.num_pages, 16, 1, 64, fill=0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k, v, sp, cu = wl.append_batch(w, [0], [40], device="cuda")
    nk.kv_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), k, v, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_PAGE
    # rows of the valid pages still landed where the oracle puts them
    opool = oracle.new_pool(w.num_pages, 16, 1, 64)
    assert oracle.kv_append(opool, w.num_pages, 16, 1, 64, bt, sp, cu, k.cpu(), v.cpu()) == 16
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    status.zero_()
    k1, v1, _, cu1 = wl.append_batch(w, [0], [1], device="cuda")
    nk.kv_append(pool, bt.cuda(), torch.tensor([3 * 16], dtype=torch.int32, device="cuda"), cu1.cuda(), k1, v1,
                 status=status)        # position past the block table (max_pages = 3)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_POS


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_flags_bad_context(impl):
    w = small("badctx", 2, 2, 4, 2, 64, 16, [40, 30], seed=2, num_pages=8)
    c = build(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx = torch.tensor([1, 30], dtype=torch.int32, device="cuda")   # ctx < T for sequence 0
    out = run_decode(c, impl, ctx=ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_CTX
    ref = oracle.paged_attention(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu, [40, 30], c.q_cpu, w.T, w.Hq,
                                 w.sm_scale)
    compare(out[1], ref[1], "valid sequence next to a bad one")


def test_decode_step_flags_bad_context_before_its_wait():
    """nk_decode_step's split kernel checks the context lengths before it
    waits for the step's append; a bad length is flagged, the other
    sequence is still right, and the append's rows land bit-exactly."""
    T = 2
    w = small("badctx_step", 2, T, 24, 4, 256, 64, [300, 700], seed=8, num_pages=20)
    c = build(w)
    hist_lens = [L - T for L in w.ctx_lens]
    # history is the whole context minus the step's T rows; re-append those rows through decode_step
    k, v, sp, cu = wl.append_batch(w, hist_lens, [T, T], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx = torch.tensor([1, w.ctx_lens[1]], dtype=torch.int32, device="cuda")  # ctx < T for sequence 0
    out = nk.decode_step(c.pool, c.bt, sp.cuda(), cu.cuda(), k, v, c.q, ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_CTX
    assert np.array_equal(gpu_pool_bytes(c), c.opool), "rows re-appended by decode_step differ"
    compare(out[1], oracle_attention_full(c)[1], "valid sequence next to a bad one")


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_ignores_garbage_past_context(impl):
    """Slots past ctx_len hold 0xFF bytes (NaN scales, -1 codes); the output
    must not see them."""
    w = small("garbage", 3, 4, 24, 4, 256, 64, [70, 129, 5], seed=9, num_pages=9)
    c = build(w, fill=0xFF)
    assert np.array_equal(gpu_pool_bytes(c), c.opool)
    ref = oracle_attention_full(c)
    out = run_decode(c, impl)
    torch.cuda.synchronize()
    compare(out, ref, "garbage past ctx")


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_page_permutation_bit_identical(impl):
    w = small("perm", 2, 4, 24, 4, 256, 64, [300, 1000], seed=4, num_pages=30)
    c = build(w)
    a = run_decode(c, impl)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(1))
    cb = nk.kv_chunk_bytes(w.P, w.D) * w.Hkv
    moved = torch.empty_like(c.pool.storage).view(w.num_pages, cb)
    moved[perm.cuda()] = c.pool.storage.view(w.num_pages, cb)
    pool2 = nk.KVPool(moved.view(-1), w.num_pages, w.P, w.Hkv, w.D)
    bt2 = torch.where(c.bt_cpu >= 0, perm[c.bt_cpu.clamp(min=0).long()].to(torch.int32), c.bt_cpu).cuda()
    fn = nk.paged_decode_attn if impl == "mma" else nk.paged_decode_attn_simt
    b = fn(pool2, c.q, bt2, c.ctx, w.sm_scale, w.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_combine_matches_oracle():
    rng = np.random.default_rng(21)
    for S, R, D in [(1, 5, 64), (4, 33, 256), (7, 8, 128), (16, 100, 256)]:
        po = rng.standard_normal((S, R, D)).astype(np.float32)
        pl = (rng.standard_normal((S, R)) * 5).astype(np.float32)
        pl[rng.random((S, R)) < 0.2] = -np.inf
        if S > 1:
            pl[:, 0] = -np.inf                    # an all-empty row -> zeros
        out = nk.attn_combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda())
        torch.cuda.synchronize()
        ref = oracle.combine(po, pl)
        got = out.to(torch.float64).cpu().numpy()
        exp = oracle.bits_to_double(oracle.round_bf16(ref))
        # one bf16 ulp at most (fp32 accumulation vs fp64)
        assert np.all(np.abs(got - exp) <= np.abs(exp) * 2.0 ** -7 + 1e-30)
        assert np.linalg.norm(got - exp) <= 1e-3 * max(np.linalg.norm(exp), 1e-30)
