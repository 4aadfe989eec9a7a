"""Pins of the oracle's append, paged attention and combine (CPU only).

Each test checks the oracle against something it does not share code with:
torch's scaled_dot_product_attention (fp64, CPU) on the unquantized inputs in
the lossless case, closed forms, invariances the definition implies, and the
byte count the "NInfer-3090" README prints for the INT8 format. Chosen so that
a dropped term, a wrong index (page, slot, group, head), an off-by-one in the
causal limit or a transposed operand fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def lossless_rows(rng, n, H, D, exp_range=(-3, 3)):
    """bf16 rows whose 64-groups quantize without loss: x = q * 2^-e with
    integer q in [-127, 127] and one |q| = 127 per group, so s = 2^-e exactly."""
    q = rng.integers(-127, 128, size=(n, H, D // 64, 64))
    pos = rng.integers(0, 64, size=(n, H, D // 64))
    sgn = rng.choice([-1, 1], size=(n, H, D // 64))
    np.put_along_axis(q, pos[..., None], (127 * sgn)[..., None], axis=-1)
    e = rng.integers(exp_range[0], exp_range[1] + 1, size=(n, H, D // 64, 1))
    x = (q * np.exp2(-e.astype(np.float64))).reshape(n, H, D)
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float64), torch.from_numpy(x)), "lossless construction must be exact in bf16"
    return t


class Case:
    """A paged cache filled through the oracle's own append."""

    def __init__(self, rng, B, T, Hq, Hkv, D, P, lens, lossless=True, spare_pages=3, fill=0, k_exp=(-3, 3)):
        self.B, self.T, self.Hq, self.Hkv, self.D, self.P = B, T, Hq, Hkv, D, P
        self.lens = list(lens)
        need = [(L + P - 1) // P for L in lens]
        self.num_pages = sum(need) + spare_pages
        self.max_pages = max(need) + 1
        perm = rng.permutation(self.num_pages)
        self.bt = np.full((B, self.max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            self.bt[b, :need[b]] = perm[off:off + need[b]]
            off += need[b]
        self.pool = oracle.new_pool(self.num_pages, P, Hkv, D, fill=fill)
        self.k, self.v = [], []
        for b in range(B):
            if lossless:
                k, v = lossless_rows(rng, lens[b], Hkv, D, k_exp), lossless_rows(rng, lens[b], Hkv, D)
            else:
                k = torch.from_numpy(rng.standard_normal((lens[b], Hkv, D))).to(torch.bfloat16)
                v = torch.from_numpy(rng.standard_normal((lens[b], Hkv, D))).to(torch.bfloat16)
            self.k.append(k)
            self.v.append(v)
        k = torch.cat(self.k)
        v = torch.cat(self.v)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        rc = oracle.kv_append(self.pool, self.num_pages, P, Hkv, D, self.bt, np.zeros(B, np.int32), cu, k, v)
        assert rc == 0
        self.q = torch.from_numpy(rng.standard_normal((B, T, Hq, D))).to(torch.bfloat16)
        self.scale = 1.0 / np.sqrt(D)

    def attention(self, **kw):
        return oracle.paged_attention(self.pool, self.num_pages, self.P, self.Hkv, self.D, self.bt,
                                      np.array(self.lens, np.int32), self.q, self.T, self.Hq, self.scale, **kw)

    def scores_max_weight(self):
        """Median over rows of the largest softmax weight (unquantized inputs, torch fp64)."""
        tops = []
        for b in range(self.B):
            L = self.lens[b]
            G = self.Hq // self.Hkv
            q = self.q[b].to(torch.float64)                                  # [T, Hq, D]
            k = self.k[b].to(torch.float64).repeat_interleave(G, dim=1)     # [L, Hq, D]
            z = torch.einsum("thd,lhd->thl", q, k) * self.scale
            n = torch.arange(L)[None, None, :]
            t = torch.arange(self.T)[:, None, None]
            z = z.masked_fill(n > (L - self.T + t), float("-inf"))
            tops.append(torch.softmax(z, dim=-1).amax(dim=-1).flatten())
        return float(torch.cat(tops).median())

    def sdpa(self):
        """Dense causal GQA attention on the unquantized rows (torch, fp64)."""
        outs = []
        for b in range(self.B):
            L = self.lens[b]
            q = self.q[b].to(torch.float64).permute(1, 0, 2)[None]           # [1, Hq, T, D]
            k = self.k[b].to(torch.float64).permute(1, 0, 2)[None]           # [1, Hkv, L, D]
            v = self.v[b].to(torch.float64).permute(1, 0, 2)[None]
            n = torch.arange(L)[None, :]
            t = torch.arange(self.T)[:, None]
            mask = n <= (L - self.T + t)                                    # [T, L]
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=self.scale, enable_gqa=True)
            outs.append(o[0].permute(1, 0, 2))                              # [T, Hq, D]
        return torch.stack(outs).numpy()


# Key scales 2^-e: e in [-3, 3] gives keys up to +-1016 and near one-hot
# softmax rows (a dominant key per row: index and selection errors show);
# e in [5, 8] gives keys within +-4 and scores of order 1, so many keys weigh
# in every row (normalization and weighting errors show).
@pytest.mark.parametrize("k_exp", [(-3, 3), (5, 8)], ids=["peaked", "temperate"])
@pytest.mark.parametrize("B,T,Hq,Hkv,D,P,lens", [
    (1, 1, 2, 1, 64, 16, [256]),
    (2, 1, 6, 2, 128, 16, [37, 130]),
    (3, 4, 12, 2, 64, 32, [4, 70, 129]),
    (2, 8, 8, 4, 256, 16, [8, 45]),
    (1, 3, 24, 4, 256, 64, [200]),
])
def test_lossless_equals_dense_sdpa(B, T, Hq, Hkv, D, P, lens, k_exp):
    rng = np.random.default_rng(B * 100 + T)
    c = Case(rng, B, T, Hq, Hkv, D, P, lens, k_exp=k_exp)
    if k_exp[0] > 0:
        # the softmax really is spread: the largest weight of a row is well below 1
        s = c.scores_max_weight()
        assert s < 0.5, s
    np.testing.assert_allclose(c.attention(), c.sdpa(), rtol=1e-12, atol=1e-12)


def test_constant_values_give_that_value():
    """All visible V rows equal -> every output row equals it (weights sum to 1)."""
    rng = np.random.default_rng(7)
    c = Case(rng, 2, 4, 4, 2, 64, 16, [33, 50])
    row = lossless_rows(rng, 1, 2, 64)
    for b in range(2):
        c.v[b] = row.expand(c.lens[b], 2, 64).contiguous()
    cu = np.concatenate([[0], np.cumsum(c.lens)]).astype(np.int32)
    oracle.kv_append(c.pool, c.num_pages, 16, 2, 64, c.bt, np.zeros(2, np.int32), cu, torch.cat(c.k), torch.cat(c.v))
    out = c.attention()
    expect = row.to(torch.float64).numpy()[0]  # [Hkv][D]
    for i in range(4):
        np.testing.assert_allclose(out[:, :, i, :], np.broadcast_to(expect[i // 2], out[:, :, i, :].shape),
                                   rtol=1e-13, atol=1e-15)


def test_equal_keys_average_visible_values():
    """All keys equal -> uniform softmax -> mean of the visible V rows."""
    rng = np.random.default_rng(8)
    L, T = 40, 4
    c = Case(rng, 1, T, 2, 1, 64, 16, [L])
    krow = lossless_rows(rng, 1, 1, 64)
    c.k[0] = krow.expand(L, 1, 64).contiguous()
    oracle.kv_append(c.pool, c.num_pages, 16, 1, 64, c.bt, np.zeros(1, np.int32), np.array([0, L], np.int32),
                     c.k[0], c.v[0])
    out = c.attention()
    v = c.v[0].to(torch.float64).numpy()[:, 0, :]
    for t in range(T):
        np.testing.assert_allclose(out[0, t, 0], v[: L - T + t + 1].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(9)
    L = 50
    c = Case(rng, 1, 1, 1, 1, 64, 16, [L])
    c.q = torch.zeros((1, 1, 1, 64), dtype=torch.bfloat16)
    c.q[0, 0, 0, 0] = 64.0
    k = torch.zeros((L, 1, 64), dtype=torch.bfloat16)
    k[:, 0, 1] = 1.0                      # non-zero groups everywhere (scale 1/127)
    k[17, 0, 0] = 64.0                    # key 17 scores 64*64/8 = 512 above the rest
    c.k[0] = k
    oracle.kv_append(c.pool, c.num_pages, 16, 1, 64, c.bt, np.zeros(1, np.int32), np.array([0, L], np.int32),
                     k, c.v[0])
    out = c.attention()
    np.testing.assert_allclose(out[0, 0, 0], c.v[0][17, 0].to(torch.float64).numpy(), rtol=1e-14, atol=1e-14)


def test_causal_column_equals_shorter_context():
    """Column t of a T-token verify over L keys == T=1 decode over L-T+t+1 keys."""
    rng = np.random.default_rng(10)
    L, T, Hq, Hkv, D, P = 77, 5, 6, 2, 128, 16
    c = Case(rng, 1, T, Hq, Hkv, D, P, [L], lossless=False)
    full = c.attention()
    for t in range(T):
        q1 = c.q[:, t:t + 1].contiguous()
        ref = oracle.paged_attention(c.pool, c.num_pages, P, Hkv, D, c.bt, np.array([L - T + t + 1], np.int32),
                                     q1, 1, Hq, c.scale)
        np.testing.assert_array_equal(full[0, t], ref[0, 0])


def test_masked_and_stale_slots_do_not_matter():
    """Garbage (including NaN bytes) in slots past the causal limit and past
    ctx_len leaves the output bit-identical."""
    rng = np.random.default_rng(12)
    L, T, P = 45, 4, 16
    c = Case(rng, 1, T, 4, 2, 64, P, [L], lossless=False)
    ref = c.attention()
    kc, ks, vc, vs = oracle.chunk_view(c.pool, c.num_pages, P, 2, 64)
    cb = oracle.chunk_bytes(P, 64)
    # overwrite everything from position L-T+1 on with garbage, except key
    # positions that some column still sees (n <= L-1 for t = T-1): only
    # positions >= L are never seen; positions L-T+1.. L-1 are seen by later
    # columns, so perturb only what column 0 cannot see and check column 0.
    last_page = c.bt[0, (L - 1) // P]
    raw = c.pool.reshape(c.num_pages, 2, cb)
    for slot in range(L % P, P):           # slots >= L in the last page
        for h in range(2):
            raw[last_page, h, slot * 64:(slot + 1) * 64] = rng.integers(0, 256, 64, dtype=np.uint8)
            off = P * 64 + slot * 4
            raw[last_page, h, off:off + 4] = np.frombuffer(np.float32(np.nan).tobytes(), np.uint8)
            off2 = 2 * P * 64 + P * 4 + slot * 4
            raw[last_page, h, off2:off2 + 4] = np.frombuffer(np.float32(np.nan).tobytes(), np.uint8)
    np.testing.assert_array_equal(c.attention(), ref)
    # now perturb keys L-T+1 .. L-1 (visible only to later columns): column 0 unchanged
    pert = c.pool.copy()
    rawp = pert.reshape(c.num_pages, 2, cb)
    for n in range(L - T + 1, L):
        pg, slot = c.bt[0, n // P], n % P
        for h in range(2):
            rawp[pg, h, slot * 64:(slot + 1) * 64] = rng.integers(0, 256, 64, dtype=np.uint8)
    out = oracle.paged_attention(pert, c.num_pages, P, 2, 64, c.bt, np.array([L], np.int32), c.q, T, 4, c.scale)
    np.testing.assert_array_equal(out[0, 0], ref[0, 0])
    assert not np.array_equal(out[0, T - 1], ref[0, T - 1])


def test_physical_page_permutation_is_invisible():
    rng = np.random.default_rng(13)
    P, H, D = 16, 2, 64
    c = Case(rng, 2, 2, 4, H, D, P, [70, 33], lossless=False)
    ref = c.attention()
    cb = oracle.chunk_bytes(P, D)
    perm = rng.permutation(c.num_pages)               # new_page = perm[old_page]
    raw = c.pool.reshape(c.num_pages, H, cb)
    moved = np.empty_like(raw)
    moved[perm] = raw
    bt2 = np.where(c.bt >= 0, perm[np.maximum(c.bt, 0)], -1).astype(np.int32)
    out = oracle.paged_attention(moved.reshape(-1), c.num_pages, P, H, D, bt2, np.array(c.lens, np.int32), c.q,
                                 c.T, c.Hq, c.scale)
    np.testing.assert_array_equal(out, ref)


def test_split_then_combine_equals_unsplit():
    rng = np.random.default_rng(14)
    L, T, Hq, Hkv, D, P = 300, 3, 4, 2, 128, 32
    c = Case(rng, 1, T, Hq, Hkv, D, P, [L], lossless=False)
    full = c.attention()
    for trial in range(5):
        S = int(rng.integers(1, 7))
        cuts = np.sort(rng.choice(np.arange(1, L), S - 1, replace=False)) if S > 1 else np.array([], int)
        bounds = np.concatenate([[0], cuts, [L]]).astype(int)
        rows = T * Hq
        po = np.zeros((S, rows, D), np.float32)
        pl = np.zeros((S, rows), np.float32)
        po64 = np.zeros((S, rows, D))
        pl64 = np.zeros((S, rows))
        for s in range(S):
            for t in range(T):
                for i in range(Hq):
                    o, lse = oracle.attention_row(c.pool, c.num_pages, P, Hkv, D, c.bt, [L], c.q, T, Hq, c.scale,
                                                  0, t, i, int(bounds[s]), int(bounds[s + 1]))
                    po64[s, t * Hq + i], pl64[s, t * Hq + i] = o, lse
        # merge in fp64 directly (closed form) and through oracle.combine (fp32 inputs)
        m = pl64.max(axis=0)
        w = np.where(np.isfinite(pl64), np.exp(pl64 - m), 0.0)
        merged = (w[..., None] * po64).sum(0) / w.sum(0)[:, None]
        np.testing.assert_allclose(merged.reshape(T, Hq, D), full[0], rtol=1e-11, atol=1e-13)
        po[:], pl[:] = po64, pl64
        comb = oracle.combine(po, pl)
        np.testing.assert_allclose(comb.reshape(T, Hq, D), full[0], rtol=2e-6, atol=1e-7)


def test_combine_closed_forms():
    rng = np.random.default_rng(15)
    po = rng.standard_normal((3, 5, 64)).astype(np.float32)
    # single partial -> itself
    np.testing.assert_array_equal(oracle.combine(po[:1], np.zeros((1, 5), np.float32)), po[0].astype(np.float64))
    # equal LSEs -> plain mean
    np.testing.assert_allclose(oracle.combine(po, np.full((3, 5), 2.5, np.float32)),
                               po.astype(np.float64).mean(0), rtol=1e-12)
    # -inf partials carry no weight
    pl = np.array([[0.0] * 5, [-np.inf] * 5, [np.log(3.0)] * 5], np.float32)
    exp = (po[0].astype(np.float64) * 1 + po[2].astype(np.float64) * 3.0000001) / 4.0000001
    np.testing.assert_allclose(oracle.combine(po, pl), exp, rtol=1e-6)
    # all empty -> zeros
    np.testing.assert_array_equal(oracle.combine(po, np.full((3, 5), -np.inf, np.float32)), np.zeros((5, 64)))
    # large LSEs (exp would overflow without the max shift): weights 1 : 3
    pl = np.array([[1000.0] * 5, [-np.inf] * 5, [1000.0 + np.log(3.0)] * 5], np.float32)
    w2 = np.exp(np.float64(pl[2, 0]) - np.float64(pl[0, 0]))
    exp = (po[0].astype(np.float64) + po[2].astype(np.float64) * w2) / (1 + w2)
    np.testing.assert_allclose(oracle.combine(po, pl), exp, rtol=1e-12)


def test_append_in_pieces_equals_append_at_once():
    rng = np.random.default_rng(16)
    P, H, D, L = 16, 2, 128, 90
    c = Case(rng, 1, 1, 2, H, D, P, [L], lossless=False)
    pool2 = oracle.new_pool(c.num_pages, P, H, D)
    k, v = c.k[0], c.v[0]
    pos = 0
    for n in [1, 15, 3, 33, 38]:
        rc = oracle.kv_append(pool2, c.num_pages, P, H, D, c.bt, np.array([pos], np.int32),
                              np.array([0, n], np.int32), k[pos:pos + n].contiguous(), v[pos:pos + n].contiguous())
        assert rc == 0
        pos += n
    np.testing.assert_array_equal(pool2, c.pool)


def test_append_writes_each_group_where_the_table_says():
    rng = np.random.default_rng(17)
    P, H, D = 16, 3, 128
    c = Case(rng, 2, 1, 3, H, D, P, [21, 40], lossless=False)
    kc, ks, vc, vs = oracle.chunk_view(c.pool, c.num_pages, P, H, D)
    for b in range(2):
        for n in range(c.lens[b]):
            pg, slot = c.bt[b, n // P], n % P
            for h in range(H):
                for g in range(D // 64):
                    q, s = oracle.quantize_group(bits(c.k[b][n, h, g * 64:(g + 1) * 64]))
                    np.testing.assert_array_equal(kc[pg, h, slot, g * 64:(g + 1) * 64], q)
                    assert ks[pg, h, slot, g] == np.float32(s)
                    q, s = oracle.quantize_group(bits(c.v[b][n, h, g * 64:(g + 1) * 64]))
                    np.testing.assert_array_equal(vc[pg, h, slot, g * 64:(g + 1) * 64], q)
                    assert vs[pg, h, slot, g] == np.float32(s)


def test_append_rejects_out_of_range_positions():
    rng = np.random.default_rng(18)
    c = Case(rng, 1, 1, 1, 1, 64, 16, [20])
    k = torch.zeros((1, 1, 64), dtype=torch.bfloat16)
    before = c.pool.copy()
    assert oracle.kv_append(c.pool, c.num_pages, 16, 1, 64, c.bt, np.array([c.max_pages * 16], np.int32),
                            np.array([0, 1], np.int32), k, k) == 1
    bt = c.bt.copy()
    bt[0, 0] = c.num_pages  # page id outside the pool
    assert oracle.kv_append(c.pool, c.num_pages, 16, 1, 64, bt, np.array([0], np.int32),
                            np.array([0, 1], np.int32), k, k) == 1
    np.testing.assert_array_equal(c.pool, before)


def test_bytes_per_token_matches_page():
    vals = {}
    with open(os.path.join(GOLDEN, "bytes_per_token.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    P, D = 64, vals["head_dim"]
    per_token_head = oracle.chunk_bytes(P, D) // P
    codes = 2 * D
    scales_here = per_token_head - codes
    groups = 2 * (D // 64)
    assert scales_here == groups * vals["scale_bytes_here"]
    page_fmt = (codes + groups * vals["scale_bytes_page"]) * vals["layers"] * vals["kv_heads"]
    assert page_fmt == vals["page_bytes_per_token_int8"]
    assert per_token_head * vals["layers"] * vals["kv_heads"] == vals["bytes_per_token_here"]
