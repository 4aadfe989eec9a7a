"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant below is oracle.c with one plausible mistake planted in it: a
dropped term, a wrong sign, rounding rule or bound, a wrong or transposed
index (page, slot, group, head, query row), a swapped operand. Every mutant is
compiled into a library of its own, and the oracle pins (the quantizer,
attention, rk8v4 and formats test files) run against it in a child process; each mutant must be
caught, i.e. make at least one pin fail, while the unaltered source, built the
same way, passes all of them. The mistakes are planted in copies in a
temporary directory: oracle.c itself is never changed.

Mistakes that cannot change any result are not listed, with the reason:
  * the clamp to [-127, 127]: fp32(x / s) with |x| <= absmax and
    s = fp32(absmax / 127) is at most 127 (1 + 2^-24) < 127.5, so the clamp
    never acts and no input can tell a different clamp apart;
  * the rk8v4 value clamp to [-7, 7], for the same reason (fp32(x / s) with
    s = RN_fp16(absmax / 7) is at most 7 (1 + 2^-11) < 7.5);
  * subtracting a different finite reference than the maximum in the softmax
    or in the combine (the weights' ratios do not depend on it);
  * skipping the empty partials in the combine (exp(-inf) = 0 already).
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_quantize.py", "tests/test_oracle_attention.py", "tests/test_oracle_rk8v4.py",
        "tests/test_oracle_formats.py"]

ROT_LINE = ("for (int j = 0; j < GROUP; ++j) rk_add_term(acc, x[j], __builtin_popcount((unsigned)(r & j)) & 1);\n"
            "    y[r] = rk_round_fp32(acc);")
# the whole transform in fp32 butterflies, every add rounded, then x 1/8
FP32_BUTTERFLIES = ("float t[GROUP];\n    for (int i = 0; i < GROUP; ++i) t[i] = (float)oracle_bf16_to_double(x[i]);\n"
                    "    for (int h = {first}; {cond}; {step})\n"
                    "      for (int i = 0; i < GROUP; ++i)\n"
                    "        if ((i & h) == 0) {{ const float a = t[i], b = t[i + h]; t[i] = a + b; t[i + h] = a - b; }}\n"
                    "    y[r] = t[r] * 0.125f; (void)acc;")

# (name, section, [(text in oracle.c, replacement), ...]); each text occurs
# exactly once in its section of oracle.c: "int8" (the INT8 group-64 format,
# the combine and the shared helpers), "rk8v4" (from its banner to the next),
# "formats" (the INT8 layout with fp16 scales and the bf16 layout).
MUTANTS = [
    # quantizer
    ("scale divides by 128", "int8", [("(float)(a / 127.0)", "(float)(a / 128.0)")]),
    ("zero group gets scale 1/2", "int8", [("(a == 0.0) ? 1.0f", "(a == 0.0) ? 0.5f")]),
    ("absmax without the absolute value", "int8",
     [("double v = fabs(oracle_bf16_to_double(x[i]));", "double v = oracle_bf16_to_double(x[i]);")]),
    ("quotient not rounded to fp32", "int8",
     [("float r = (float)(oracle_bf16_to_double(x[i]) / (double)s);",
       "double r = oracle_bf16_to_double(x[i]) / (double)s;")]),
    ("ties away from zero", "int8", [("double k = nearbyint((double)r);", "double k = round((double)r);")]),
    ("truncation instead of rounding", "int8", [("double k = nearbyint((double)r);", "double k = trunc((double)r);")]),
    # bf16 helpers
    ("bf16 with 9 significant bits", "int8",
     [("r = ldexp(nearbyint(ldexp(m, 8)), e - 8);", "r = ldexp(nearbyint(ldexp(m, 9)), e - 9);")]),
    ("bf16 rounding truncates", "int8",
     [("r = ldexp(nearbyint(ldexp(m, 8)), e - 8);", "r = ldexp(trunc(ldexp(m, 8)), e - 8);")]),
    ("bf16 subnormal quantum 2^-132", "int8",
     [("r = nearbyint(ldexp(x, 133)) * ldexp(1.0, -133);", "r = nearbyint(ldexp(x, 132)) * ldexp(1.0, -132);")]),
    ("bf16 widening drops the sign", "int8",
     [("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)(bits & 0x7fffu) << 16;")]),
    # pool layout
    ("K and V scale arrays swapped", "int8",
     [("c.ks = (float*)(base + (size_t)P * D);",
       "c.ks = (float*)(base + 2 * (size_t)P * D + (size_t)P * g * sizeof(float));"),
      ("c.vs = (float*)(base + 2 * (size_t)P * D + (size_t)P * g * sizeof(float));",
       "c.vs = (float*)(base + (size_t)P * D);")]),
    ("chunk index misses the head stride", "int8",
     [("((size_t)page * num_kv_heads + head)", "((size_t)page + head)")]),
    # append
    ("append slot off by one", "int8", [("int slot = (int)(pos % P);", "int slot = (int)((pos + 1) % P);")]),
    ("append ignores the block table", "int8",
     [("int page = block_table[(size_t)b * max_pages + pos / P];", "int page = (int)(pos / P);")]),
    ("append assigns boundary rows to the wrong sequence", "int8",
     [("while (b + 1 <= B && cu_new[b + 1] <= j) ++b;", "while (b + 1 < B && cu_new[b + 1] < j) ++b;")]),
    ("append reads K rows head-major", "int8",
     [("const uint16_t* krow = k + ((size_t)j * H + h) * D;",
       "const uint16_t* krow = k + ((size_t)h * total + j) * D;")]),
    ("append quantizes V from K", "int8",
     [("oracle_quantize_group(vrow + gr * GROUP", "oracle_quantize_group(krow + gr * GROUP")]),
    # attention
    ("q-head i reads kv-head i mod Hkv", "int8", [("const int h = i / G;", "const int h = i % H;")]),
    ("no causal mask among the T columns", "int8", [("const long last = L - T + t;", "const long last = L - 1;")]),
    ("causal limit one key short", "int8", [("const long last = L - T + t;", "const long last = L - T + t - 1;")]),
    ("query rows read head-major", "int8",
     [("const uint16_t* qrow = q + (((size_t)b * T + t) * Hq + i) * D;",
       "const uint16_t* qrow = q + (((size_t)b * Hq + i) * T + t) * D;")]),
    ("softmax scale dropped", "int8", [("z[n - n0] = sm_scale * dot;", "z[n - n0] = dot;")]),
    ("K pages read without the block table", "int8",
     [("int page = block_table[(size_t)b * max_pages + n / P];\n    if (page < 0",
       "int page = (int)(n / P);\n    if (page < 0")]),
    ("K group scale indexed by channel mod groups", "int8",
     [("(double)c.ks[(size_t)slot * g + ch / GROUP];", "(double)c.ks[(size_t)slot * g + ch % g];")]),
    ("V dequantized with the K scales", "int8",
     [("(double)c.vs[(size_t)slot * g + ch / GROUP]", "(double)c.ks[(size_t)slot * g + ch / GROUP]")]),
    ("V channels of a pair transposed", "int8",
     [("((double)c.vc[(size_t)slot * D + ch]", "((double)c.vc[(size_t)slot * D + (ch ^ 1)]")]),
    ("softmax weights without the max shift but LSE with it", "int8",
     [("double w = exp(z[n - n0] - m);", "double w = exp(z[n - n0]);")]),
    ("softmax sum counts keys", "int8", [("l += w;", "l += 1.0;")]),
    ("output not normalized", "int8", [("for (int ch = 0; ch < D; ++ch) o[ch] /= l;", "")]),
    ("LSE without the max", "int8", [("*lse = m + log(l);", "*lse = log(l);")]),
    # combine
    ("combine weight with the wrong sign", "int8", [("double w = exp(ls - m);", "double w = exp(m - ls);")]),
    ("combine not normalized", "int8", [("for (int c = 0; c < D; ++c) o[c] /= wsum;", "")]),
    ("combine partials read row-major", "int8",
     [("part_o[((size_t)s * R + r) * D + c]", "part_o[((size_t)r * S + s) * D + c]")]),
    # rk8v4: fp16 helpers, rotation, quantizers, layout, attention
    ("fp16 with 10 significant bits", "rk8v4",
     [("r = ldexp(nearbyint(ldexp(a, 11 - e)), e - 11);", "r = ldexp(nearbyint(ldexp(a, 10 - e)), e - 10);")]),
    ("fp16 subnormal quantum 2^-23", "rk8v4",
     [("r = nearbyint(ldexp(a, 24)) * ldexp(1.0, -24);", "r = nearbyint(ldexp(a, 23)) * ldexp(1.0, -23);")]),
    ("rotation without the 1/8", "rk8v4", [("ldexp(mant, low - 136)", "ldexp(mant, low - 133)")]),
    ("rotation sign from r | j", "rk8v4",
     [("rk_add_term(acc, x[j], __builtin_popcount((unsigned)(r & j)) & 1)",
       "rk_add_term(acc, x[j], __builtin_popcount((unsigned)(r | j)) & 1)")]),
    ("rotation as fp32 butterflies over bits 0..5", "rk8v4", [(ROT_LINE, FP32_BUTTERFLIES.format(first="1", step="h <<= 1", cond="h < GROUP"))]),
    ("rotation as fp32 butterflies over bits 5..0", "rk8v4", [(ROT_LINE, FP32_BUTTERFLIES.format(first="GROUP / 2", step="h >>= 1", cond="h >= 1"))]),
    ("rotation summed in fp64, then rounded", "rk8v4",
     [(ROT_LINE, "double s = 0.0;\n    for (int j = 0; j < GROUP; ++j) { const double v = oracle_bf16_to_double(x[j]); "
                 "s += (__builtin_popcount((unsigned)(r & j)) & 1) ? -v : v; }\n    y[r] = (float)(s / 8.0);")]),
    ("rotation rounding ignores the sticky bits", "rk8v4",
     [("if (guard && (sticky || fmod(mant, 2.0) == 1.0)) mant += 1.0;", "if (guard && fmod(mant, 2.0) == 1.0) mant += 1.0;")]),
    ("rotation rounds ties away from zero", "rk8v4",
     [("if (guard && (sticky || fmod(mant, 2.0) == 1.0)) mant += 1.0;", "if (guard) mant += 1.0;")]),
    ("rotation carries truncate instead of floor", "rk8v4", [("if (acc[k] - c * 65536 < 0) c -= 1;", "")]),
    ("keys stored unrotated", "rk8v4",
     [("oracle_rk_rotate64(krow + gr * GROUP, y);",
       "for (int ii = 0; ii < GROUP; ++ii) y[ii] = (float)oracle_bf16_to_double(krow[gr * GROUP + ii]);")]),
    ("key scale divides by 128", "rk8v4", [("rk_scale_bits(a, 127.0)", "rk_scale_bits(a, 128.0)")]),
    ("value scale divides by 8", "rk8v4", [("rk_scale_bits(a, 7.0)", "rk_scale_bits(a, 8.0)")]),
    ("scale below the fp16 range kept tiny", "rk8v4", [("if ((sb & 0x7fff) == 0) sb = 0x3c00;", "if ((sb & 0x7fff) == 0) sb = 0x0001;")]),
    ("scale past the fp16 range left infinite", "rk8v4", [("else if ((sb & 0x7fff) == 0x7c00) sb = 0x7bff;", "")]),
    ("value nibbles in the other order", "rk8v4",
     [("packed[j] = (uint8_t)((q[2 * j] & 0xf) | ((q[2 * j + 1] & 0xf) << 4));",
       "packed[j] = (uint8_t)((q[2 * j + 1] & 0xf) | ((q[2 * j] & 0xf) << 4));")]),
    ("value groups written 32 bytes apart", "rk8v4",
     [("c.vc + (size_t)slot * (D / 2) + gr * (VGROUP / 2))", "c.vc + (size_t)slot * (D / 2) + gr * VGROUP)")]),
    ("value nibbles read without sign extension", "rk8v4", [("return n >= 8 ? n - 16 : n;", "return n;")]),
    ("query not rotated", "rk8v4", [("qr[g0 + r] = acc / 8.0;", "qr[g0 + r] = oracle_bf16_to_double(qrow[g0 + r]);")]),
    ("query rotation sign from r | j", "rk8v4",
     [("(__builtin_popcount((unsigned)(r & jj)) & 1) ? -x : x", "(__builtin_popcount((unsigned)(r | jj)) & 1) ? -x : x")]),
    ("key scale indexed per 32 channels", "rk8v4",
     [("oracle_f16_to_double(c.ks[(size_t)slot * (D / GROUP) + ch / GROUP])",
       "oracle_f16_to_double(c.ks[(size_t)slot * (D / GROUP) + ch / VGROUP])")]),
    ("value scale indexed per 64 channels", "rk8v4",
     [("c.vs[(size_t)slot * (D / VGROUP) + ch / VGROUP]", "c.vs[(size_t)slot * (D / VGROUP) + ch / GROUP]")]),
    # rk8v4: the same attention and append logic as the INT8 section, planted there too
    ("rk8v4: q-head i reads kv-head i mod Hkv", "rk8v4", [("const int h = i / G;", "const int h = i % H;")]),
    ("rk8v4: causal limit one key short", "rk8v4",
     [("const long last = L - T + t;", "const long last = L - T + t - 1;")]),
    ("rk8v4: append slot off by one", "rk8v4", [("int slot = (int)(pos % P);", "int slot = (int)((pos + 1) % P);")]),
    ("rk8v4: append ignores the block table", "rk8v4",
     [("int page = block_table[(size_t)b * max_pages + pos / P];", "int page = (int)(pos / P);")]),
    ("rk8v4: K pages read without the block table", "rk8v4",
     [("int page = block_table[(size_t)b * max_pages + n / P];\n    if (page < 0",
       "int page = (int)(n / P);\n    if (page < 0")]),
    ("rk8v4: softmax scale dropped", "rk8v4", [("z[n - n0] = sm_scale * dot;", "z[n - n0] = dot;")]),
    ("rk8v4: output not normalized", "rk8v4", [("for (int ch = 0; ch < D; ++ch) o[ch] /= l;", "")]),
    ("rk8v4: LSE without the max", "rk8v4", [("*lse = m + log(l);", "*lse = log(l);")]),
    # the INT8 layout with fp16 scales and the bf16 layout
    ("int8_f16: scales indexed per 32 channels", "formats",
     [("((size_t)slot * g + ch / GROUP) * 2, 2);", "((size_t)slot * g + ch / 32) * 2, 2);")]),
    ("int8_f16: V codes read from the K half", "formats",
     [("const uint8_t* part = base + (want_v ? half : 0);", "const uint8_t* part = base;")]),
    ("int8_f16: V scale stored over the K scale", "formats",
     [("memcpy(base + half + (size_t)P * D + ((size_t)slot * g + gr) * 2, &sv, 2);",
       "memcpy(base + (size_t)P * D + ((size_t)slot * g + gr) * 2, &sv, 2);")]),
    ("bf16: V read from the K rows", "formats",
     [("memcpy(&bits, base + (want_v ? (size_t)P * D * 2 : 0) + ((size_t)slot * D + ch) * 2, 2);",
       "memcpy(&bits, base + ((size_t)slot * D + ch) * 2, 2);")]),
    ("formats: q-head i reads kv-head i mod Hkv", "formats", [("const int h = i / G;", "const int h = i % H;")]),
    ("formats: causal limit one key short", "formats",
     [("const long n1 = L - T + t + 1;", "const long n1 = L - T + t;")]),
    ("formats: output not normalized", "formats", [("for (int ch = 0; ch < D; ++ch) o[ch] /= l;", "")]),
]

RUNNER = (
    "import sys, oracle, pytest\n"
    "oracle.use_library(sys.argv[1])\n"
    "sys.exit(pytest.main(['-x', '-q', '-rf', '-p', 'no:cacheprovider', '-W', 'ignore'] + sys.argv[2:]))\n"
)


def _source() -> str:
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        return f.read()


BANNERS = {
    "rk8v4": "/* ===========================================================================\n * rk8v4",
    "formats": "/* ===========================================================================\n * The pages' own INT8",
}


def _mutate(src: str, section: str, edits) -> str:
    cuts = [0, src.index(BANNERS["rk8v4"]), src.index(BANNERS["formats"]), len(src)]
    k = {"int8": 0, "rk8v4": 1, "formats": 2}[section]
    head, part, tail = src[:cuts[k]], src[cuts[k]:cuts[k + 1]], src[cuts[k + 1]:]
    for old, new in edits:
        assert part.count(old) == 1, f"mutation anchor not unique or missing in {section}: {old!r}"
        part = part.replace(old, new)
    return head + part + tail


def _build_and_run(src: str, workdir: str, tag: str):
    c_path = os.path.join(workdir, f"{tag}.c")
    so_path = os.path.join(workdir, f"{tag}.so")
    with open(c_path, "w") as f:
        f.write(src)
    inc = os.path.join(ROOT, "oracle")
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", inc, "-o", so_path, c_path, "-lm"], check=True,
                   capture_output=True)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-c", RUNNER, so_path, *PINS], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    failed = [ln.split(" ")[1] for ln in r.stdout.splitlines() if ln.startswith("FAILED ")]
    return r.returncode, failed, r.stdout[-2000:] + r.stderr[-2000:]


def test_every_mutant_fails_a_pin(tmp_path):
    src = _source()
    jobs = [("unaltered", src)] + [(f"m{i:02d}", _mutate(src, sec, edits)) for i, (_, sec, edits) in enumerate(MUTANTS)]
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda j: _build_and_run(j[1], str(tmp_path), j[0]), jobs))
    rc0, failed0, log0 = results[0]
    assert rc0 == 0, f"the unaltered oracle must pass every pin:\n{log0}"
    survivors, crashed = [], []
    for (name, _, _), (rc, failed, log) in zip(MUTANTS, results[1:]):
        if rc == 0:
            survivors.append(name)
        elif rc != 1 or not failed:
            crashed.append(f"{name}: exit {rc}\n{log}")
    assert not crashed, "mutants must be caught by a failing pin, not by a crash:\n" + "\n".join(crashed)
    assert not survivors, f"mutants no pin catches: {survivors}"


@pytest.mark.parametrize("name,section,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutation_anchors_exist(name, section, edits):
    """Each planted mistake still applies to the current oracle.c."""
    _mutate(_source(), section, edits)
