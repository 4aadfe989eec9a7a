"""Pins of the oracle's quantizer and bf16 helpers (CPU only).

The oracle's quantizer computes in fp64 and rounds once to fp32; these tests
check it against routes that share none of its code: numpy's IEEE float32
division and round-half-even, hand-derived golden groups, invariants that
follow from the definition, and an exhaustive sweep over every finite bf16
value. Rule: s = fp32(absmax / 127) (1 if absmax = 0),
q = clamp(round_half_even(fp32(x / s)), -127, 127)  (INT8 group-64 KV,
"NInfer" README capability list; rounding rule as read by this library).
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits_to_bf16(x32: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp32 values that are exactly bf16."""
    b = np.asarray(x32, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value is not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def numpy_reference(x_bits: np.ndarray):
    """Independent route: numpy float32 IEEE division, np.rint (half to even)."""
    x = oracle.bits_to_double(x_bits).astype(np.float32)
    a = np.max(np.abs(x))
    s = np.float32(1.0) if a == 0 else np.float32(a) / np.float32(127.0)
    r = (x / s).astype(np.float32)
    q = np.clip(np.rint(r), -127, 127).astype(np.int8)
    return q, np.float32(s)


def random_group(rng, scale=1.0, outliers=0):
    x = (rng.standard_normal(64) * scale).astype(np.float32)
    if outliers:
        idx = rng.choice(64, outliers, replace=False)
        x[idx] *= 8.0
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("seed", range(6))
def test_matches_numpy_float32(seed):
    rng = np.random.default_rng(seed)
    for i in range(400):
        scale = float(10.0 ** rng.uniform(-30, 30))
        xb = random_group(rng, scale, outliers=int(rng.integers(0, 5)))
        q, s = oracle.quantize_group(xb)
        q2, s2 = numpy_reference(xb)
        assert np.float32(s) == s2
        np.testing.assert_array_equal(q, q2)


def test_invariants():
    rng = np.random.default_rng(11)
    for _ in range(2000):
        xb = random_group(rng, float(10.0 ** rng.uniform(-3, 3)))
        q, s = oracle.quantize_group(xb)
        x = oracle.bits_to_double(xb)
        a = np.max(np.abs(x))
        assert np.all(np.abs(q.astype(int)) <= 127)
        if a > 0:
            assert np.max(np.abs(q.astype(int))) == 127  # the absmax element maps to +-127
            # |x - q s| <= s (1/2 + 2^-17): the 1/2 of rounding to an integer plus
            # the fp32 rounding of x/s (|x/s| <= 127.00001)
            assert np.all(np.abs(x - q.astype(np.float64) * s) <= s * (0.5 + 2.0 ** -17))
        nz = q != 0
        assert np.all(np.sign(q[nz]) == np.sign(x[nz]))


def test_zero_group():
    q, s = oracle.quantize_group(np.zeros(64, dtype=np.uint16))
    assert s == 1.0 and not q.any()
    # negative zeros too
    q, s = oracle.quantize_group(np.full(64, 0x8000, dtype=np.uint16))
    assert s == 1.0 and not q.any()


def load_cases():
    cases = []
    with open(os.path.join(GOLDEN, "quantize_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line.startswith("case"):
                continue
            body = line[4:]
            xs, s, qs = (part.strip() for part in body.split("|"))
            x = np.zeros(64, dtype=np.float32)
            for tok in xs.split():
                i, v = tok.split(":")
                x[int(i)] = float(v)
            q = np.zeros(64, dtype=np.int8)
            for tok in qs.split():
                i, v = tok.split(":")
                q[int(i)] = int(v)
            cases.append((x, np.float32(float(s)), q))
    return cases


@pytest.mark.parametrize("case", range(4))
def test_golden_cases(case):
    x, s_exp, q_exp = load_cases()[case]
    q, s = oracle.quantize_group(f32_bits_to_bf16(x))
    assert np.float32(s) == s_exp
    np.testing.assert_array_equal(q, q_exp)


@pytest.mark.parametrize("absmax", [1.0, 3.0, 0.1, 200.0, 1e-20])
def test_exhaustive_bf16(absmax):
    """Every finite bf16 value x with |x| <= absmax, placed in a group whose
    absmax element is fixed: the oracle's code equals numpy's float32 route."""
    allb = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bits_to_double(allb)
    am = float(torch.tensor(absmax, dtype=torch.float32).to(torch.bfloat16).float())
    keep = np.isfinite(vals) & (np.abs(vals) <= am)
    xs = allb[keep]
    amb = f32_bits_to_bf16(np.array([am], dtype=np.float32))[0]
    # one group per 63 values plus the absmax element
    for i in range(0, xs.size, 63):
        chunk = xs[i:i + 63]
        grp = np.concatenate([np.array([amb], dtype=np.uint16), chunk,
                              np.zeros(63 - chunk.size, dtype=np.uint16)])
        q, s = oracle.quantize_group(grp)
        q2, s2 = numpy_reference(grp)
        assert np.float32(s) == s2
        np.testing.assert_array_equal(q, q2)


def test_double_to_bf16_against_torch():
    """Doubles that are exact fp32 values round to bf16 like torch's fp32->bf16 (RNE)."""
    rng = np.random.default_rng(5)
    x32 = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-35, 35, 200000)).astype(np.float32)
    ours = oracle.round_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_double_to_bf16_ties_and_specials():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even -> 1.0
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is the midpoint between 1+2^-7 and 1+2^-6: ties to even -> 1+2^-6 (0x3F82)
    assert oracle.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the midpoint rounds up (a double, not an fp32 value)
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.double_to_bf16(0.0) == 0x0000
    assert oracle.double_to_bf16(-0.0) == 0x8000
    assert oracle.double_to_bf16(1e300) == 0x7F80
    assert oracle.double_to_bf16(-1e300) == 0xFF80
    # smallest bf16 subnormal is 2^-133
    assert oracle.double_to_bf16(2.0 ** -133) == 0x0001
    assert oracle.double_to_bf16(2.0 ** -134) == 0x0000  # tie to even (zero)
    assert oracle.double_to_bf16(2.0 ** -134 + 2.0 ** -160) == 0x0001


def test_bf16_widening_exact():
    allb = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(allb.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    for i in range(0, 1 << 16, 4099):
        a, b = oracle.bf16_to_double(int(allb[i])), ref[i]
        assert (a == b) or (np.isnan(a) and np.isnan(b))
