"""The MXFP4 decode's f16x2 powers of two, made by one rounding conversion
of binary32 powers of two, equal the f16 bits built field by field (normal,
subnormal, zero) for every pair of exponents in [-300, 0]: the check program
compiles the library's own device helpers and compares all pairs on the
GPU."""
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "nvfp4_kv_cache_bd_gb300", "csrc")


def test_f16x2_pow2_matches_the_field_by_field_bits():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "pow2_check")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", CSRC,
                        os.path.join(HERE, "pow2_check.cu"), "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    words = out.split()
    assert words[0] == "checked" and int(words[1]) == 301 * 301, out
    assert words[2] == "mismatches" and int(words[3]) == 0, out
