"""The rk8v4 kernels' scale rounding, replayed on the CPU.

tests/rk_scale_check.c compares the kernel's route for a group scale (the
IEEE fp32 quotient max|x| / c rounded again to fp16) with the oracle's (the
fp64 quotient rounded once to fp16) for every positive bf16 value-group
maximum (c = 7) and every fp32 key-group maximum of 71 binary exponents
(c = 127): 5.96 * 10^8 cases, which must agree one for one. The scales
themselves follow the "NInfer-3090" README, "RotorQuant KV (rk8v4)" (fp16
scales, 4-bit values over 32 channels, INT8 keys over 64).
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_kernel_scale_route_equals_single_rounding(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "rk_scale_check"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-std=c11", "-o", str(exe),
                    os.path.join(HERE, "rk_scale_check.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout
    tested, bad = out.stdout.split()[-3], out.stdout.split()[-1]
    assert int(bad) == 0 and int(tested) > 5 * 10 ** 8, out.stdout
