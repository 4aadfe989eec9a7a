"""The append kernel's division-free quotient, replayed on the CPU.

tests/quotient_check.c repeats the kernel's fp32 steps (y = RN(1/s),
q0 = RN(x*y), one fma remainder, one fma correction, magic-number rounding) and
compares each int8 code with the IEEE quotient rounded half to even, for every
bf16 element of every bf16 group maximum over the exponents that matter. The
quantization rule itself is the "NInfer" README's INT8 group-64 format.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_refined_quotient_matches_ieee_division(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "quotient_check"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-std=c11", "-o", str(exe),
                    os.path.join(HERE, "quotient_check.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout
    tested, bad = out.stdout.split()[-3], out.stdout.split()[-1]
    assert int(bad) == 0 and int(tested) > 10 ** 8, out.stdout
