"""GPU parity of the rk8v4 format against the oracle.

rk8v4 ("NInfer-3090" README, "RotorQuant KV (rk8v4)"): rotated INT8 group-64
keys and 4-bit group-32 values with fp16 scales. The append must reproduce
the oracle's pool bytes exactly (codes, scales, untouched bytes); attention
must meet the same tolerance as the INT8 path against the oracle's fp64
result rounded to bf16. Inputs are the seeded synthetic workloads; the oracle
never sees a value computed by the CUDA path (attention is compared on the
pool the oracle itself appended, copied to the GPU).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import Built, compare

pytestmark = pytest.mark.gpu


def build_rk(w, fill=0, chunk=16384):
    """History of every sequence appended through both paths in the same chunks."""
    c = Built()
    c.w = w
    c.bt_cpu = wl.block_table(w)
    c.bt = c.bt_cpu.cuda()
    c.ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    c.pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, fill=fill, fmt="rk8v4")
    c.opool = oracle.rk_new_pool(w.num_pages, w.P, w.Hkv, w.D, fill=fill)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(w.B):
        pos = 0
        while pos < w.ctx_lens[b]:
            n = min(chunk, w.ctx_lens[b] - pos)
            k, v = wl.kv_rows(w, b, pos, n)
            cu = torch.tensor([0, n], dtype=torch.int32)
            nk.rk8v4_append(c.pool, c.bt[b:b + 1].contiguous(), torch.tensor([pos], dtype=torch.int32, device="cuda"),
                            cu.cuda(), k.cuda(), v.cuda(), status=status)
            assert oracle.rk_append(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu[b:b + 1], [pos], cu, k, v) == 0
            pos += n
    torch.cuda.synchronize()
    c.status = int(status.item())
    c.q = wl.queries(w).cuda()
    c.q_cpu = c.q.cpu()
    return c


def oracle_out(c, ctx=None):
    w = c.w
    return oracle.rk_paged_attention(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu,
                                     w.ctx_lens if ctx is None else ctx, c.q_cpu, w.T, w.Hq, w.sm_scale)


def use_oracle_pool(c):
    c.pool.storage.copy_(torch.from_numpy(c.opool).cuda())


CASES = {
    # name: (B, T, Hq, Hkv, D, P, ctx_lens)
    "d64_p16": (2, 1, 2, 1, 64, 16, [37, 300]),
    "d128_g3_t3": (3, 3, 6, 2, 128, 32, [3, 64, 517]),
    "d256_g6_t1": (2, 1, 24, 4, 256, 64, [130, 1900]),
    "d256_g6_t4": (3, 4, 24, 4, 256, 64, [4, 700, 2049]),
    "d256_g8_t2": (2, 2, 16, 2, 256, 16, [90, 333]),
    "d256_g6_t12": (2, 12, 24, 4, 256, 64, [12, 640]),  # two column chunks
    "d64_g1_t16": (1, 16, 4, 4, 64, 16, [400]),
    "d256_p256": (2, 2, 12, 2, 256, 256, [300, 1100]),  # pages too large for the staged kernel's ring
}


def case(name, seed=5, fill=0):
    B, T, Hq, Hkv, D, P, lens = CASES[name]
    w = wl.custom(f"rk_{name}", B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=seed,
                  outlier_channels=2 if D >= 128 else 0, outlier_scale=8.0)
    return build_rk(w, fill=fill)


@pytest.mark.parametrize("name", list(CASES))
def test_append_bit_exact(name):
    c = case(name, fill=0x5A)
    assert c.status == 0
    got = c.pool.storage.cpu().numpy()
    diff = np.flatnonzero(got != c.opool)
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"


def test_append_ragged_batch_in_one_call():
    """One call with unaligned starts, an empty sequence and page-crossing runs."""
    P, D, H = 16, 128, 2
    starts, lens = [5, 0, 31, 16], [40, 0, 3, 17]
    num_pages = 24
    rng = np.random.default_rng(9)
    bt = torch.from_numpy(rng.permutation(num_pages)[:4 * 6].reshape(4, 6).astype(np.int32))
    k = (torch.randn((sum(lens), H, D)) * 3).to(torch.bfloat16)
    v = torch.randn((sum(lens), H, D)).to(torch.bfloat16)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int32)
    pool = nk.KVPool.empty(num_pages, P, H, D, fill=0x33, fmt="rk8v4")
    opool = oracle.rk_new_pool(num_pages, P, H, D, fill=0x33)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.rk8v4_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda(), status=status)
    assert oracle.rk_append(opool, num_pages, P, H, D, bt, sp, cu, k, v) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pool.storage.cpu().numpy(), opool)


def wide_key_rows(n, H, D, seed):
    """Key rows whose 64-channel groups span far more than 39 binades (values
    from 2^-133 to 2^120, two clusters 2^100 apart, exact cancellations), so
    that the append rotates them by its exact integer route; the rest of the
    rows are ordinary groups (fp64 route)."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, H, D // 64, 64))
    kind = rng.integers(0, 4, size=(n, H, D // 64))
    wide = 2.0 ** rng.uniform(-133, 120, size=k.shape)
    clusters = np.where(rng.random(k.shape) < 0.5, 2.0 ** 40, 2.0 ** -60)
    k = np.where((kind == 1)[..., None], k * wide, k)
    k = np.where((kind == 2)[..., None], k * clusters, k)
    # kind 3: channel pairs (0, 1) equal, so half of the outputs cancel them exactly
    k3 = k.copy()
    k3[..., 0] = 2.0 ** 70
    k3[..., 1] = 2.0 ** 70
    k3[..., 2:] *= 2.0 ** -40
    k = np.where((kind == 3)[..., None], k3, k)
    return torch.from_numpy(k.reshape(n, H, D)).to(torch.bfloat16)


@pytest.mark.parametrize("n", [256, 512])
def test_append_wide_exponent_key_groups_bit_exact(n):
    """Both routes of the key rotation against the oracle's exact rotation
    rounded once: codes and scales bit for bit; saturated scales may flag.
    256 rows (2,048 key groups) take the warp-per-group kernel of small
    appends, 512 rows the thread-per-item kernel."""
    H, D, P = 2, 256, 64
    k = wide_key_rows(n, H, D, seed=21)
    v = torch.randn((n, H, D)).to(torch.bfloat16)
    num_pages = n // P
    bt = torch.arange(num_pages, dtype=torch.int32)[None].contiguous()
    cu = torch.tensor([0, n], dtype=torch.int32)
    sp = torch.tensor([0], dtype=torch.int32)
    pool = nk.KVPool.empty(num_pages, P, H, D, fill=0x11, fmt="rk8v4")
    opool = oracle.rk_new_pool(num_pages, P, H, D, fill=0x11)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.rk8v4_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda(), status=status)
    assert oracle.rk_append(opool, num_pages, P, H, D, bt, sp, cu, k, v) == 0
    torch.cuda.synchronize()
    assert int(status.item()) & ~0x10 == 0
    got = pool.storage.cpu().numpy()
    diff = np.flatnonzero(got != opool)
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"


def sweep_rows():
    """K and V rows whose group maxima sweep the scale's range: every positive
    finite bf16 value below 458,000 is the absmax of one value group (its
    scale stays within fp16, down to the groups whose scale underflows to 0
    and is stored as 1); key groups span magnitudes 1e-30 .. 1e5."""
    allb = np.arange(1 << 15, dtype=np.uint32).astype(np.uint16)  # sign bit clear
    vals = oracle.bits_to_double(allb)
    amax = allb[np.isfinite(vals) & (vals > 0) & (vals < 458000.0)]
    H, D = 4, 256
    per_row = H * D // 32
    rows = (amax.size + per_row - 1) // per_row
    rng = np.random.default_rng(12)
    frac = rng.uniform(-1, 1, size=(rows * per_row, 32))
    am = np.concatenate([amax, np.full(rows * per_row - amax.size, 0x3F80, np.uint16)])
    am64 = oracle.bits_to_double(am)
    v = torch.from_numpy(frac * am64[:, None]).to(torch.bfloat16)
    v = v.view(torch.int16)
    v[:, 0] = torch.from_numpy(am.view(np.int16))  # the absmax element itself
    v = v.view(torch.bfloat16).reshape(rows, H, D)
    mag = 10.0 ** rng.uniform(-30, 5, size=(rows, H, D // 64, 1))
    k = torch.from_numpy(rng.standard_normal((rows, H, D // 64, 64)) * mag).to(torch.bfloat16).reshape(rows, H, D)
    return k, v


@pytest.mark.parametrize("rows_per_call", [0, 64])
def test_append_scale_sweep_bit_exact(rows_per_call):
    """The whole sweep in one call (thread-per-item kernel) or in calls of 64
    rows (1,024 key groups each: the warp-per-group kernel)."""
    k, v = sweep_rows()
    n, H, D = k.shape
    P = 64
    num_pages = (n + P - 1) // P
    bt = torch.arange(num_pages, dtype=torch.int32).flip(0)[None].contiguous()
    pool = nk.KVPool.empty(num_pages, P, H, D, fill=0, fmt="rk8v4")
    opool = oracle.rk_new_pool(num_pages, P, H, D, fill=0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = rows_per_call or n
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        sp, cu = torch.tensor([r0], dtype=torch.int32), torch.tensor([0, r1 - r0], dtype=torch.int32)
        kk, vv = k[r0:r1].contiguous(), v[r0:r1].contiguous()
        nk.rk8v4_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), kk.cuda(), vv.cuda(), status=status)
        assert oracle.rk_append(opool, num_pages, P, H, D, bt, sp, cu, kk, vv) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = pool.storage.cpu().numpy()
    diff = np.flatnonzero(got != opool)
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_append_saturating_scales_flag_range():
    """Groups past the fp16 scale range: scales saturate at 65504 exactly as in
    the oracle, codes clamp, and NK_DEVFLAG_RANGE is raised; zero groups get
    scale 1."""
    H, D, P = 1, 64, 16
    k = torch.zeros((3, H, D))
    v = torch.zeros((3, H, D))
    k[0, 0, 5] = 3e9    # rotated absmax 3.75e8 > 127 * 65504
    v[1, 0, 40] = -1e6  # absmax 1e6 > 7 * 65504
    k[2, 0, :] = 1.0    # rotated: one entry 8, the rest 0
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    bt = torch.tensor([[0]], dtype=torch.int32)
    sp, cu = torch.zeros(1, dtype=torch.int32), torch.tensor([0, 3], dtype=torch.int32)
    pool = nk.KVPool.empty(1, P, H, D, fill=0, fmt="rk8v4")
    opool = oracle.rk_new_pool(1, P, H, D, fill=0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.rk8v4_append(pool, bt.cuda(), sp.cuda(), cu.cuda(), k.cuda(), v.cuda(), status=status)
    assert oracle.rk_append(opool, 1, P, H, D, bt, sp, cu, k, v) == 0
    torch.cuda.synchronize()
    assert int(status.item()) & 0x10
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    kc, ks, vc, vs = oracle.rk_chunk_view(opool, 1, P, H, D)
    assert ks[0, 0, 0, 0] == 0x7BFF and vs[0, 0, 1, 1] == 0x7BFF
    assert vs[0, 0, 0, 0] == 0x3C00 and ks[0, 0, 1, 0] == 0x3C00


def test_append_flags_bad_pages_and_positions():
    H, D, P = 1, 64, 16
    k = torch.randn((2, H, D)).to(torch.bfloat16)
    bt = torch.tensor([[7, 0]], dtype=torch.int32)  # page 7 of a 2-page pool
    pool = nk.KVPool.empty(2, P, H, D, fill=0, fmt="rk8v4")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.rk8v4_append(pool, bt.cuda(), torch.tensor([0], dtype=torch.int32, device="cuda"),
                    torch.tensor([0, 2], dtype=torch.int32, device="cuda"), k.cuda(), k.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_PAGE
    status.zero_()
    nk.rk8v4_append(pool, bt.cuda(), torch.tensor([32], dtype=torch.int32, device="cuda"),  # past 2 pages
                    torch.tensor([0, 2], dtype=torch.int32, device="cuda"), k.cuda(), k.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_POS
    assert not pool.storage.any(), "nothing may be written for a skipped row"


@pytest.mark.parametrize("num_ctas", [0, 1, 37, 300])
@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name, num_ctas):
    c = case(name)
    use_oracle_pool(c)
    w = c.w
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.rk8v4_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=num_ctas, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, oracle_out(c), f"{name} n={num_ctas}")


def test_decode_is_deterministic_and_ignores_garbage_past_context():
    c = case("d256_g6_t4", fill=0)
    use_oracle_pool(c)
    w = c.w
    a = nk.rk8v4_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    b = nk.rk8v4_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    # every byte of every slot past its sequence's context becomes 0xFF (NaN scales)
    st = c.pool.storage.view(w.num_pages, w.Hkv, -1).clone()
    lay = nk.rk8v4_chunk_bytes(w.P, w.D)
    assert st.shape[-1] == lay
    P, D = w.P, w.D
    ks, vc, vs = P * D, P * D + P * (D // 64) * 2, P * D + P * (D // 64) * 2 + P * D // 2
    for bi, L in enumerate(w.ctx_lens):
        last_page = (L - 1) // P
        page = int(c.bt_cpu[bi, last_page])
        s0 = L - last_page * P
        if s0 == P:
            continue
        st[page, :, s0 * D:P * D] = 0xFF
        st[page, :, ks + s0 * (D // 64) * 2:vc] = 0xFF
        st[page, :, vc + s0 * (D // 2):vs] = 0xFF
        st[page, :, vs + s0 * (D // 32) * 2:] = 0xFF
    c.pool.storage.copy_(st.view(-1))
    g = nk.rk8v4_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a, g)


def test_decode_flags_bad_context_and_pages():
    c = case("d64_p16")
    use_oracle_pool(c)
    w = c.w
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_ctx = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    nk.rk8v4_decode_attn(c.pool, c.q, c.bt, bad_ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_CTX
    status.zero_()
    bt = c.bt.clone()
    bt[1, 3] = w.num_pages + 5
    nk.rk8v4_decode_attn(c.pool, c.q, bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_PAGE


def test_full_size_c1_rk8v4():
    """c1_rk8v4 (c1_decode's inputs, rk8v4 format), in the launch
    configuration the benchmark times: the append of the whole 32,768-token
    history bit-exact, every output row within tolerance."""
    w = wl.make("c1_rk8v4")
    c = build_rk(w)
    assert c.status == 0
    got = c.pool.storage.cpu().numpy()
    assert np.array_equal(got, c.opool), "pool bytes differ"
    out = nk.rk8v4_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    compare(out, oracle_out(c), "c1_rk8v4")
