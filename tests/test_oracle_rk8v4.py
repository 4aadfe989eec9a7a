"""Pins of the oracle's rk8v4 format (CPU only).

rk8v4 ("NInfer-3090" README, "RotorQuant KV (rk8v4)"): keys rotated by the
64-point Hadamard transform and stored as INT8 group-64 codes, values as
signed 4-bit group-32 codes, fp16 scales. The oracle is checked against
routes that share none of its code: numpy's float16/float32 arithmetic for the
scales and codes, scipy's Hadamard matrix for the rotation, the page's
bytes-per-token figure, and torch's fp64 scaled_dot_product_attention on
inputs that the format stores without loss (rotated key groups with at most
two non-zero entries, values q * 2^-e with |q| <= 7), plus closed forms and
invariances of attention.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
H64 = scipy.linalg.hadamard(64).astype(np.float64)  # Sylvester order


def to_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16(x) -> np.ndarray:
    """Round to bf16 and back (fp64)."""
    return oracle.bits_to_double(to_bits(x))


# ---------------------------------------------------------------- fp16 helpers

def test_f16_widening_every_pattern():
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = allb.view(np.float16).astype(np.float64)
    ours = np.array([oracle.f16_to_double(int(b)) for b in allb])
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_f16_rounding_against_numpy():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(60000) * 10.0 ** rng.uniform(-9, 6, 60000)
    # ties and the edges of the range
    x = np.concatenate([x, [1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24,
                            65504.0, 65519.99, 65520.0, 1e9, -65520.0, 6.1e-5, 0.0, -0.0]])
    ours = np.array([oracle.double_to_f16(v) for v in x], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------- rotation

def test_rotation_is_scaled_hadamard_on_exact_inputs():
    """Small integers: every partial sum is exact, so R x = H64 x / 8 exactly."""
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = rng.integers(-100, 101, 64).astype(np.float64) * 2.0 ** int(rng.integers(-20, 20))
        y = oracle.rk_rotate64(to_bits(x))
        np.testing.assert_array_equal(y.astype(np.float64), H64 @ x / 8.0)


def exponent_span(x) -> int:
    """Binades between the smallest and the largest non-zero |x| (bf16)."""
    e = np.floor(np.log2(np.abs(x[x != 0])))
    return int(e.max() - e.min()) if e.size else 0


def test_rotation_rounds_once_on_general_inputs():
    """bf16 inputs of mixed magnitude within 30 binades: each partial sum of
    H64 x is an integer multiple of the smallest input's quantum below 2^53
    of it, so scipy's Hadamard matrix times x in fp64 is exact, / 8 is exact,
    and one rounding to float32 is the definition. Bit for bit equal -- a
    rotation that rounds in between (fp32 butterflies in any order) differs
    on most of these groups."""
    rng = np.random.default_rng(5)
    differs_from_fp32_butterflies = 0
    for _ in range(400):
        x = bf16(rng.choice([-1.0, 1.0], 64) * rng.uniform(1.0, 2.0, 64) * 2.0 ** rng.uniform(-15, 15, 64))
        x[rng.random(64) < 0.05] = 0.0
        assert exponent_span(x) <= 38
        y = oracle.rk_rotate64(to_bits(x))
        ref = (H64 @ x / 8.0).astype(np.float32)
        np.testing.assert_array_equal(y, ref)
        t = x.astype(np.float32)
        h = 1
        while h < 64:
            for i in range(64):
                if i & h == 0:
                    t[i], t[i + h] = t[i] + t[i + h], t[i] - t[i + h]
            h <<= 1
        differs_from_fp32_butterflies += int(np.any(t * np.float32(0.125) != ref))
    assert differs_from_fp32_butterflies > 300


def fraction_to_f32(r: Fraction) -> np.float32:
    """Round a rational to float32: nearest, ties to even, overflow to inf."""
    if r == 0:
        return np.float32(0.0)
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    q = max(e, -126) - 23                      # quantum of float32 at |r|
    n = round(a / Fraction(2) ** q)            # Fraction.__round__: half to even
    mag = n * Fraction(2) ** q
    if mag >= Fraction(2) ** 128:
        v = np.inf
    else:
        v = float(n) * 2.0 ** q                # exact: n < 2^25, q >= -149
    return np.float32(v if r > 0 else -v)


def rotate_exact(x_bits) -> np.ndarray:
    """H64 x / 8 in exact rational arithmetic, rounded once to float32."""
    xs = [Fraction(float(v)) for v in oracle.bits_to_double(np.asarray(x_bits, dtype=np.uint16))]
    return np.array([fraction_to_f32(sum((xs[j] if H64[r, j] > 0 else -xs[j]) for j in range(64)) / 8)
                     for r in range(64)], dtype=np.float32)


def wide_groups():
    """Groups whose partial sums are not exact in fp64: exponent spans of up
    to 250 binades, exact cancellation of the large terms, bf16 subnormals,
    sums at an fp32 tie with a tiny term deciding it, float32-subnormal and
    overflowing results."""
    rng = np.random.default_rng(11)
    gs = []
    for _ in range(40):  # random magnitudes over the whole bf16 range
        gs.append(bf16(rng.standard_normal(64) * 2.0 ** rng.uniform(-130, 125, 64)))
    for _ in range(20):  # two clusters far apart
        x = rng.standard_normal(64) * 2.0 ** 60
        x[rng.random(64) < 0.5] *= 2.0 ** -110
        gs.append(bf16(x))
    big = 2.0 ** 90
    x = np.zeros(64)
    x[0], x[1] = big, big           # H rows with popcount(r & 1) = 1 cancel the large terms exactly
    x[2] = 2.0 ** -100
    x[5] = -3 * 2.0 ** -120
    gs.append(x)
    x = np.zeros(64)                # an fp32 tie (1 + 2^-24) decided by a term 2^-100 below it
    x[0] = 8 * (1.0 + 2.0 ** -7)    # 1 + 2^-7 and 2^-24: bf16, and the group sums to a tie
    x[1] = 8 * 2.0 ** -17
    x[2] = 8 * 2.0 ** -24
    x[3] = 8 * 2.0 ** -100
    gs.append(bf16(x))
    x[3] = -x[3]
    gs.append(bf16(x))
    x = np.zeros(64)                # exact ties with nothing below: to even, down then up
    x[0], x[2] = 8 * (1.0 + 2.0 ** -7), 8 * 2.0 ** -24
    gs.append(bf16(x))
    x = np.zeros(64)
    x[0], x[1], x[2] = 8 * (1.0 + 2.0 ** -7), 8 * 2.0 ** -23, 8 * 2.0 ** -24
    gs.append(bf16(x))
    gs.append(bf16(np.full(64, 2.0 ** -133)))                 # bf16 subnormals: fp32-subnormal results
    gs.append(bf16(rng.choice([-1, 1], 64) * 2.0 ** -130))
    gs.append(bf16(np.full(64, 3.0e38)))                      # the first output overflows float32
    gs.append(bf16(np.r_[np.full(32, 3.0e38), np.full(32, -3.0e38)]))
    return gs


def test_rotation_rounds_once_on_wide_and_degenerate_groups():
    for i, x in enumerate(wide_groups()):
        bits = to_bits(x)
        y = oracle.rk_rotate64(bits)
        ref = rotate_exact(bits)
        same = (y == ref) | (np.isnan(y) & np.isnan(ref))
        assert same.all(), f"group {i}: outputs {np.nonzero(~same)[0][:8]} differ"


def test_rotation_tie_cases_round_as_the_definition_says():
    """The hand-built tie: the exact first output is 1 + 2^-24 + 2^-17 .. with
    a 2^-100 term; with the tiny term positive it rounds up, negative down."""
    gs = wide_groups()
    up, down, even_dn, even_up = gs[-8], gs[-7], gs[-6], gs[-5]
    y_up, y_dn = oracle.rk_rotate64(to_bits(up))[0], oracle.rk_rotate64(to_bits(down))[0]
    assert float(y_up) - float(y_dn) == 2.0 ** -23 * 2.0 ** np.floor(np.log2(float(y_dn)))
    # 1 + 2^-7 + 2^-24 is a tie whose lower neighbour is even: it stays down;
    # 1 + 2^-7 + 2^-23 + 2^-24 lies between an odd and an even one: it goes up
    assert float(oracle.rk_rotate64(to_bits(even_dn))[0]) == 1.0 + 2.0 ** -7
    assert float(oracle.rk_rotate64(to_bits(even_up))[0]) == 1.0 + 2.0 ** -7 + 2.0 ** -22


# ---------------------------------------------------------------- quantizers

def numpy_k(y):
    y = np.asarray(y, dtype=np.float32)
    a = np.float32(np.max(np.abs(y)))
    with np.errstate(over="ignore"):
        s = np.float16(a / np.float32(127.0))
    if s == 0:
        s = np.float16(1.0)
    if np.isinf(s):
        s = np.float16(65504.0)
    q = np.clip(np.rint(y / np.float32(s)), -127, 127).astype(np.int8)
    return q, int(np.array(s).view(np.uint16))


def numpy_v(xb):
    x = oracle.bits_to_double(xb).astype(np.float32)
    a = np.float32(np.max(np.abs(x)))
    with np.errstate(over="ignore"):
        s = np.float16(a / np.float32(7.0))
    if s == 0:
        s = np.float16(1.0)
    if np.isinf(s):
        s = np.float16(65504.0)
    q = np.clip(np.rint(x / np.float32(s)), -7, 7).astype(np.int64)
    return q, int(np.array(s).view(np.uint16))


def unpack(packed):
    """Independent nibble decode: element 2j = low nibble of byte j, 2j+1 = high nibble."""
    p = np.asarray(packed, dtype=np.int64)
    lo, hi = p & 0xF, p >> 4
    q = np.empty(2 * p.size, dtype=np.int64)
    q[0::2], q[1::2] = lo, hi
    return np.where(q >= 8, q - 16, q)


@pytest.mark.parametrize("seed", range(3))
def test_key_quantizer_matches_numpy(seed):
    rng = np.random.default_rng(seed)
    for _ in range(500):
        y = (rng.standard_normal(64) * 10.0 ** rng.uniform(-12, 8)).astype(np.float32)
        q, sb = oracle.rk_quantize_k(y)
        q2, sb2 = numpy_k(y)
        assert sb == sb2
        np.testing.assert_array_equal(q, q2)


@pytest.mark.parametrize("seed", range(3))
def test_value_quantizer_matches_numpy(seed):
    rng = np.random.default_rng(10 + seed)
    for _ in range(500):
        xb = to_bits(rng.standard_normal(32) * 10.0 ** rng.uniform(-12, 8))
        packed, sb = oracle.rk_quantize_v(xb)
        q2, sb2 = numpy_v(xb)
        assert sb == sb2
        np.testing.assert_array_equal(unpack(packed), q2)


@pytest.mark.parametrize("absmax", [1.0, 0.3, 448.0])
def test_value_quantizer_every_bf16(absmax):
    """Every finite bf16 value with |x| <= absmax, grouped with an absmax element."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bits_to_double(allb)
    keep = np.isfinite(vals) & (np.abs(vals) <= absmax)
    xs = allb[keep]
    amb = to_bits([absmax])[0]
    for i in range(0, xs.size, 31):
        chunk = xs[i:i + 31]
        grp = np.concatenate([[amb], chunk, np.zeros(31 - chunk.size, np.uint16)]).astype(np.uint16)
        packed, sb = oracle.rk_quantize_v(grp)
        q2, sb2 = numpy_v(grp)
        assert sb == sb2
        np.testing.assert_array_equal(unpack(packed), q2)


def test_quantizer_special_groups():
    # zero group: scale 1, codes 0
    q, sb = oracle.rk_quantize_k(np.zeros(64, np.float32))
    assert sb == 0x3C00 and not q.any()
    packed, sb = oracle.rk_quantize_v(np.zeros(32, np.uint16))
    assert sb == 0x3C00 and not packed.any()
    # absmax below the fp16 range: scale 1, codes 0
    y = np.zeros(64, np.float32)
    y[3] = 2.0 ** -40
    q, sb = oracle.rk_quantize_k(y)
    assert sb == 0x3C00 and not q.any()
    # absmax past the fp16 range: scale saturates at 65504 and the codes clamp
    y[3] = 1e8
    y[5] = -5e6
    q, sb = oracle.rk_quantize_k(y)
    assert sb == 0x7BFF and q[3] == 127 and q[5] == -76
    xb = to_bits([1e6] + [0.0] * 31)
    packed, sb = oracle.rk_quantize_v(xb)
    assert sb == 0x7BFF and unpack(packed)[0] == 7


def test_quantizer_invariants():
    rng = np.random.default_rng(21)
    for _ in range(1000):
        y = (rng.standard_normal(64) * 10.0 ** rng.uniform(-2, 2)).astype(np.float32)
        q, sb = oracle.rk_quantize_k(y)
        s = oracle.f16_to_double(sb)
        assert np.max(np.abs(q.astype(int))) == 127
        # the fp16 scale is within half an fp16 ulp of absmax / 127
        a = float(np.max(np.abs(y)))
        assert abs(s - a / 127) <= (a / 127) * 2.0 ** -11
        assert np.all(np.abs(y - q * s) <= s * (0.5 + 2.0 ** -17))
        xb = to_bits(rng.standard_normal(32) * 10.0 ** rng.uniform(-2, 2))
        packed, sb = oracle.rk_quantize_v(xb)
        s = oracle.f16_to_double(sb)
        qv = unpack(packed)
        x = oracle.bits_to_double(xb)
        assert np.max(np.abs(qv)) == 7 and np.all(np.abs(qv) <= 7)
        assert np.all(np.abs(x - qv * s) <= s * (0.5 + 2.0 ** -20))
        nz = qv != 0
        assert np.all(np.sign(qv[nz]) == np.sign(x[nz]))


# ---------------------------------------------------------------- layout and append

def test_bytes_per_token_matches_page():
    vals = {}
    with open(os.path.join(GOLDEN, "bytes_per_token.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    D = vals["head_dim"]
    per_token_head = oracle.rk_chunk_bytes(64, D) // 64
    assert per_token_head * vals["layers"] * vals["kv_heads"] == vals["page_bytes_per_token_rk8v4"]


def test_append_writes_each_group_where_the_layout_says():
    rng = np.random.default_rng(30)
    P, D, H, B = 16, 128, 2, 2
    lens = [5, 21]
    starts = [3, 0]
    num_pages = 8
    bt = np.array([[6, 1, -1], [2, 7, 0]], np.int32)
    pool = oracle.rk_new_pool(num_pages, P, H, D, fill=0xAB)
    k = rng.standard_normal((sum(lens), H, D))
    v = rng.standard_normal((sum(lens), H, D))
    kb, vb = to_bits(k).reshape(k.shape), to_bits(v).reshape(v.shape)
    cu = np.array([0, lens[0], sum(lens)], np.int32)
    assert oracle.rk_append(pool, num_pages, P, H, D, bt, np.array(starts, np.int32), cu, kb, vb) == 0
    kc, ks, vc, vs = oracle.rk_chunk_view(pool, num_pages, P, H, D)
    touched = set()
    for b in range(B):
        for j in range(lens[b]):
            row = cu[b] + j
            pos = starts[b] + j
            page, slot = bt[b, pos // P], pos % P
            touched.add((page, slot))
            for h in range(H):
                for g in range(D // 64):
                    y = oracle.rk_rotate64(kb[row, h, 64 * g:64 * g + 64])
                    q, sb = oracle.rk_quantize_k(y)
                    np.testing.assert_array_equal(kc[page, h, slot, 64 * g:64 * g + 64], q)
                    assert ks[page, h, slot, g] == sb
                for g in range(D // 32):
                    packed, sb = oracle.rk_quantize_v(vb[row, h, 32 * g:32 * g + 32])
                    np.testing.assert_array_equal(vc[page, h, slot, 16 * g:16 * g + 16], packed)
                    assert vs[page, h, slot, g] == sb
    # nothing else was written
    for page in range(num_pages):
        for slot in range(P):
            if (page, slot) not in touched:
                assert (kc[page, :, slot].view(np.uint8) == 0xAB).all()
                assert (vc[page, :, slot] == 0xAB).all()


# ---------------------------------------------------------------- attention

def lossless_keys(rng, n, H, D, e_range):
    """bf16 rows k whose rotated groups R k have at most two non-zero entries,
    +-127 * 2^-e and b * 2^-e (|b| <= 127): R k is exactly representable, its
    absmax is 127 * 2^-e, so the fp16 scale is 2^-e and the codes are exact."""
    y = np.zeros((n, H, D // 64, 64))
    e = rng.integers(e_range[0], e_range[1] + 1, size=(n, H, D // 64))
    i1 = rng.integers(0, 64, size=(n, H, D // 64))
    i2 = (i1 + rng.integers(1, 64, size=i1.shape)) % 64
    sgn = rng.choice([-1.0, 1.0], size=i1.shape)
    b2 = rng.integers(-127, 128, size=i1.shape).astype(np.float64)
    np.put_along_axis(y, i1[..., None], (127.0 * sgn)[..., None], axis=-1)
    np.put_along_axis(y, i2[..., None], b2[..., None], axis=-1)
    y *= np.exp2(-e.astype(np.float64))[..., None]
    k = np.einsum("ij,nhgj->nhgi", H64, y) / 8.0  # R = H64 / 8 is its own inverse
    k = k.reshape(n, H, D)
    assert np.array_equal(bf16(k), k), "lossless key construction must be exact in bf16"
    return torch.from_numpy(k).to(torch.bfloat16)


def lossless_values(rng, n, H, D):
    q = rng.integers(-7, 8, size=(n, H, D // 32, 32))
    pos = rng.integers(0, 32, size=(n, H, D // 32))
    np.put_along_axis(q, pos[..., None], (7 * rng.choice([-1, 1], size=pos.shape))[..., None], axis=-1)
    e = rng.integers(-4, 6, size=(n, H, D // 32, 1))
    v = (q * np.exp2(-e.astype(np.float64))).reshape(n, H, D)
    assert np.array_equal(bf16(v), v)
    return torch.from_numpy(v).to(torch.bfloat16)


class RkCase:
    def __init__(self, rng, B, T, Hq, Hkv, D, P, lens, k_exp=(-2, 2), lossless=True):
        self.B, self.T, self.Hq, self.Hkv, self.D, self.P = B, T, Hq, Hkv, D, P
        self.lens = list(lens)
        need = [(L + P - 1) // P for L in lens]
        self.num_pages = sum(need) + 2
        self.max_pages = max(need) + 1
        perm = rng.permutation(self.num_pages)
        self.bt = np.full((B, self.max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            self.bt[b, :need[b]] = perm[off:off + need[b]]
            off += need[b]
        self.pool = oracle.rk_new_pool(self.num_pages, P, Hkv, D)
        if lossless:
            self.k = [lossless_keys(rng, L, Hkv, D, k_exp) for L in lens]
            self.v = [lossless_values(rng, L, Hkv, D) for L in lens]
        else:
            self.k = [torch.from_numpy(rng.standard_normal((L, Hkv, D))).to(torch.bfloat16) for L in lens]
            self.v = [torch.from_numpy(rng.standard_normal((L, Hkv, D))).to(torch.bfloat16) for L in lens]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        assert oracle.rk_append(self.pool, self.num_pages, P, Hkv, D, self.bt, np.zeros(B, np.int32), cu,
                                torch.cat(self.k), torch.cat(self.v)) == 0
        self.q = torch.from_numpy(rng.standard_normal((B, T, Hq, D))).to(torch.bfloat16)
        self.scale = 1.0 / np.sqrt(D)

    def attention(self, **kw):
        return oracle.rk_paged_attention(self.pool, self.num_pages, self.P, self.Hkv, self.D, self.bt,
                                         np.array(self.lens, np.int32), self.q, self.T, self.Hq, self.scale, **kw)

    def sdpa(self):
        outs = []
        for b in range(self.B):
            L = self.lens[b]
            q = self.q[b].to(torch.float64).permute(1, 0, 2)[None]
            k = self.k[b].to(torch.float64).permute(1, 0, 2)[None]
            v = self.v[b].to(torch.float64).permute(1, 0, 2)[None]
            mask = torch.arange(L)[None, :] <= (L - self.T + torch.arange(self.T)[:, None])
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=self.scale, enable_gqa=True)
            outs.append(o[0].permute(1, 0, 2))
        return torch.stack(outs).numpy()


# key exponents: (-2, 2) gives rotated keys up to +-508 (one-hot softmax rows);
# (6, 9) keys within about +-2 (spread rows)
@pytest.mark.parametrize("k_exp", [(-2, 2), (6, 9)], ids=["peaked", "temperate"])
@pytest.mark.parametrize("B,T,Hq,Hkv,D,P,lens", [
    (1, 1, 2, 1, 64, 16, [100]),
    (2, 1, 6, 2, 128, 16, [37, 90]),
    (2, 4, 12, 2, 256, 32, [4, 77]),
    (1, 3, 24, 4, 256, 64, [150]),
])
def test_lossless_equals_dense_sdpa(B, T, Hq, Hkv, D, P, lens, k_exp):
    rng = np.random.default_rng(B * 100 + T + 7)
    c = RkCase(rng, B, T, Hq, Hkv, D, P, lens, k_exp=k_exp)
    np.testing.assert_allclose(c.attention(), c.sdpa(), rtol=1e-12, atol=1e-12)


def test_temperate_keys_spread_the_softmax():
    rng = np.random.default_rng(1 * 100 + 3 + 7)
    c = RkCase(rng, 1, 3, 24, 4, 256, 64, [150], k_exp=(6, 9))
    k = c.k[0].to(torch.float64).repeat_interleave(6, dim=1)
    z = torch.einsum("thd,lhd->thl", c.q[0].to(torch.float64), k) * c.scale
    assert float(torch.softmax(z, -1).amax(-1).median()) < 0.5


def test_causal_column_equals_shorter_context():
    rng = np.random.default_rng(41)
    L, T = 70, 4
    c = RkCase(rng, 1, T, 6, 2, 128, 16, [L], lossless=False)
    full = c.attention()
    for t in range(T):
        ref = oracle.rk_paged_attention(c.pool, c.num_pages, 16, 2, 128, c.bt, np.array([L - T + t + 1], np.int32),
                                        c.q[:, t:t + 1].contiguous(), 1, 6, c.scale)
        np.testing.assert_array_equal(full[0, t], ref[0, 0])


def test_split_then_combine_equals_unsplit():
    rng = np.random.default_rng(42)
    L, T, Hq, Hkv, D, P = 200, 2, 4, 2, 128, 32
    c = RkCase(rng, 1, T, Hq, Hkv, D, P, [L], lossless=False)
    full = c.attention()
    bounds = [0, 33, 64, 150, L]
    S = len(bounds) - 1
    po = np.zeros((S, T * Hq, D))
    pl = np.zeros((S, T * Hq))
    for s in range(S):
        for t in range(T):
            for i in range(Hq):
                o, lse = oracle.rk_attention_row(c.pool, c.num_pages, P, Hkv, D, c.bt, [L], c.q, T, Hq, c.scale,
                                                 0, t, i, bounds[s], bounds[s + 1])
                po[s, t * Hq + i], pl[s, t * Hq + i] = o, lse
    w = np.exp(pl - pl.max(axis=0))
    merged = (w[..., None] * po).sum(0) / w.sum(0)[:, None]
    np.testing.assert_allclose(merged.reshape(T, Hq, D), full[0], rtol=1e-11, atol=1e-13)


def test_constant_values_give_that_value():
    rng = np.random.default_rng(43)
    c = RkCase(rng, 1, 2, 4, 2, 64, 16, [40])
    row = lossless_values(rng, 1, 2, 64)
    c.v[0] = row.expand(40, 2, 64).contiguous()
    c.pool[:] = 0
    assert oracle.rk_append(c.pool, c.num_pages, 16, 2, 64, c.bt, np.zeros(1, np.int32), np.array([0, 40], np.int32),
                            c.k[0], c.v[0]) == 0
    out = c.attention()
    expect = row.to(torch.float64).numpy()[0]
    for i in range(4):
        np.testing.assert_allclose(out[0, :, i, :], np.broadcast_to(expect[i // 2], (2, 64)), rtol=1e-13, atol=0)
