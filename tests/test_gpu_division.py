"""The quantizers' division matches IEEE division at the e4m3 level on every
(amax, x) pair of bf16 inputs: built and run as a standalone CUDA program."""
import os
import re
import subprocess

import pytest

from mxfp8_precision_gemms_fp8bw_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_exhaustive(tmp_path):
    exe = str(tmp_path / "division_exhaustive")
    cmd = [build._nvcc(), *build.ARCH, "-O3", "-std=c++17", "-I" + build.CSRC,
           os.path.join(HERE, "cuda", "division_exhaustive.cu"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    m = re.search(r"checked (\d+) code_mismatches (\d+)", r.stdout)
    assert m, r.stdout + r.stderr
    checked, bad = int(m.group(1)), int(m.group(2))
    # amax over the 32640 non-negative finite bf16 patterns; for each, the
    # 2 * (pattern + 1) bf16 values x with |x| <= amax
    assert checked == 32640 * 32641, r.stdout
    assert bad == 0, r.stdout
