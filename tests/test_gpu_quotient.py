"""The quantisers compute fl32(x / s) without a division per element (two
remainder-correction steps after a correctly rounded reciprocal). This test
builds a small CUDA program around the library's own device function and
compares it with the IEEE division bit for bit on every (tile maximum, value)
pair of BF16 inputs that a quantiser tile can contain."""
import os
import subprocess

import pytest

from blockwise_fp8_linear_weight_b300 import build as lib_build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_quotient_equals_ieee_division_on_every_bf16_pair(tmp_path):
    exe = str(tmp_path / "quotient_exhaustive")
    cmd = [lib_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-prec-div=true", "-ftz=false", "-I", lib_build.CSRC,
           os.path.join(HERE, "cuda", "quotient_exhaustive.cu"), "-o", exe]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " mismatches 0 " in r.stdout
