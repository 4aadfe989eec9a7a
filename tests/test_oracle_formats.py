"""Pins of the oracle's other two layouts (CPU only): the pages' own INT8
layout with fp16 scales, and the unquantized bf16 baseline.

"NInfer-3090" README, "Choosing a KV format": int8 at 33,792 bytes per token
and bf16 at 65,536 on the 27B model (16 attention layers x 4 kv-heads, head
dim 256). Checked against: the page's byte counts; numpy's float32/float16
arithmetic for the quantizer, on random groups and on every bf16 value below
fixed group maxima; torch's fp64 scaled_dot_product_attention, exactly for
bf16 pages and on inputs the INT8 layout stores without loss (x = q * 2^-e,
|q| <= 127 with one +-127 per group, so the fp16 scale is 2^-e); and the
INT8/fp32-scale oracle where both layouts hold the same codes.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_bits(x) -> np.ndarray:
    return torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def numpy_i8h(xb):
    x = oracle.bits_to_double(xb).astype(np.float32)
    a = np.float32(np.max(np.abs(x)))
    with np.errstate(over="ignore"):
        s = np.float16(a / np.float32(127.0))
    if s == 0:
        s = np.float16(1.0)
    if np.isinf(s):
        s = np.float16(65504.0)
    q = np.clip(np.rint(x / np.float32(s)), -127, 127).astype(np.int8)
    return q, int(np.array(s).view(np.uint16))


def golden():
    vals = {}
    with open(os.path.join(GOLDEN, "bytes_per_token.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_bytes_per_token_match_the_page():
    g = golden()
    D, per = g["head_dim"], g["layers"] * g["kv_heads"]
    assert oracle.fmt_chunk_bytes("int8_f16", 64, D) // 64 * per == g["page_bytes_per_token_int8"]
    assert oracle.fmt_chunk_bytes("bf16", 64, D) // 64 * per == g["page_bytes_per_token_bf16"]


@pytest.mark.parametrize("seed", range(3))
def test_quantizer_matches_numpy(seed):
    rng = np.random.default_rng(seed)
    for _ in range(600):
        xb = to_bits(rng.standard_normal(64) * 10.0 ** rng.uniform(-12, 9))
        q, sb = oracle.i8h_quantize_group(xb)
        q2, sb2 = numpy_i8h(xb)
        assert sb == sb2
        np.testing.assert_array_equal(q, q2)


@pytest.mark.parametrize("absmax", [1.0, 0.05, 3000.0])
def test_quantizer_every_bf16(absmax):
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bits_to_double(allb)
    xs = allb[np.isfinite(vals) & (np.abs(vals) <= absmax)]
    amb = to_bits([absmax])[0]
    for i in range(0, xs.size, 63):
        chunk = xs[i:i + 63]
        grp = np.concatenate([[amb], chunk, np.zeros(63 - chunk.size, np.uint16)]).astype(np.uint16)
        q, sb = oracle.i8h_quantize_group(grp)
        q2, sb2 = numpy_i8h(grp)
        assert sb == sb2
        np.testing.assert_array_equal(q, q2)


class FmtCase:
    def __init__(self, fmt, rng, B, T, Hq, Hkv, D, P, lens, lossless=True):
        self.fmt, self.B, self.T, self.Hq, self.Hkv, self.D, self.P = fmt, B, T, Hq, Hkv, D, P
        self.lens = list(lens)
        need = [(L + P - 1) // P for L in lens]
        self.num_pages = sum(need) + 2
        perm = rng.permutation(self.num_pages)
        self.bt = np.full((B, max(need) + 1), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            self.bt[b, :need[b]] = perm[off:off + need[b]]
            off += need[b]
        self.k, self.v = [], []
        for L in lens:
            if lossless:
                q = rng.integers(-127, 128, size=(2, L, Hkv, D // 64, 64))
                pos = rng.integers(0, 64, size=(2, L, Hkv, D // 64))
                np.put_along_axis(q, pos[..., None], (127 * rng.choice([-1, 1], size=pos.shape))[..., None], axis=-1)
                e = rng.integers(-3, 9, size=(2, L, Hkv, D // 64, 1))
                x = (q * np.exp2(-e.astype(np.float64))).reshape(2, L, Hkv, D)
            else:
                x = rng.standard_normal((2, L, Hkv, D))
            t = torch.from_numpy(x).to(torch.bfloat16)
            self.k.append(t[0])
            self.v.append(t[1])
        self.pool = oracle.fmt_new_pool(fmt, self.num_pages, P, Hkv, D)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        assert oracle.fmt_append(fmt, self.pool, self.num_pages, P, Hkv, D, self.bt, np.zeros(B, np.int32), cu,
                                 torch.cat(self.k), torch.cat(self.v)) == 0
        self.q = torch.from_numpy(rng.standard_normal((B, T, Hq, D))).to(torch.bfloat16)
        self.scale = 1.0 / np.sqrt(D)

    def attention(self):
        return oracle.fmt_paged_attention(self.fmt, self.pool, self.num_pages, self.P, self.Hkv, self.D, self.bt,
                                          np.array(self.lens, np.int32), self.q, self.T, self.Hq, self.scale)

    def sdpa(self):
        outs = []
        for b in range(self.B):
            L = self.lens[b]
            q = self.q[b].to(torch.float64).permute(1, 0, 2)[None]
            k = self.k[b].to(torch.float64).permute(1, 0, 2)[None]
            v = self.v[b].to(torch.float64).permute(1, 0, 2)[None]
            mask = torch.arange(L)[None, :] <= (L - self.T + torch.arange(self.T)[:, None])
            outs.append(F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=self.scale,
                                                       enable_gqa=True)[0].permute(1, 0, 2))
        return torch.stack(outs).numpy()


SHAPES = [(1, 1, 2, 1, 64, 16, [90]), (2, 3, 6, 2, 128, 32, [3, 150]), (2, 4, 24, 4, 256, 64, [4, 130])]


@pytest.mark.parametrize("shape", SHAPES, ids=["d64", "d128_t3", "d256_t4"])
@pytest.mark.parametrize("fmt,lossless", [("int8_f16", True), ("bf16", False)], ids=["int8_f16_lossless", "bf16"])
def test_attention_equals_dense_sdpa(fmt, lossless, shape):
    B, T, Hq, Hkv, D, P, lens = shape
    c = FmtCase(fmt, np.random.default_rng(B + T), B, T, Hq, Hkv, D, P, lens, lossless=lossless)
    np.testing.assert_allclose(c.attention(), c.sdpa(), rtol=1e-12, atol=1e-12)


def test_int8_f16_equals_int8_f32_layout_on_equal_codes():
    """Where the fp16 scale equals the fp32 scale (a / 127 exactly representable
    in fp16 as well), both INT8 layouts store the same codes and give the same
    attention."""
    rng = np.random.default_rng(8)
    P, D, H, L = 16, 128, 2, 70
    c = FmtCase("int8_f16", rng, 1, 2, 4, H, D, P, [L])
    pool32 = oracle.new_pool(c.num_pages, P, H, D)
    assert oracle.kv_append(pool32, c.num_pages, P, H, D, c.bt, [0], [0, L], c.k[0], c.v[0]) == 0
    out32 = oracle.paged_attention(pool32, c.num_pages, P, H, D, c.bt, [L], c.q, 2, 4, c.scale)
    np.testing.assert_allclose(c.attention(), out32, rtol=1e-13, atol=1e-14)
