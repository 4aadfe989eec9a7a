"""The C ABI from plain C (GPU): tests/abi_step.c, a decode loop that
includes only include/nk.h and links libnk.so and the CUDA runtime, built
with the host C compiler and run. It appends a 32,767-token history, runs
220 steps of nk_decode_step_host (one sequence, T = 1, 24 q-heads over 4
kv-heads, head_dim 256), then reruns the last step through nk_decode_step on
device copies of the same inputs: every call must return NK_OK, the status
words must stay 0 and the two outputs must be identical bit for bit. The
program's JSON line (microseconds per step, host clock around each call) is
printed with the test output."""
import json
import os
import shutil
import subprocess

import pytest

from quantized_paged_kv_cache_gb300 import _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_decode_loop_in_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    assert os.path.exists(_build.LIB), "libnk.so is not built"
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    exe = str(tmp_path / "abi_step")
    libdir = os.path.dirname(_build.LIB)
    cmd = [cc, "-O2", "-Wall", "-o", exe, os.path.join(HERE, "abi_step.c"), "-I", _build.INCLUDE,
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lnk", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(run.stdout.strip())
    assert run.returncode == 0, f"abi_step exited {run.returncode}: {run.stdout} {run.stderr}"
    res = json.loads(run.stdout.strip().splitlines()[-1])
    assert res["match"] and res["finite"] and res["status"] == 0 and res["status_after_check"] == 0
