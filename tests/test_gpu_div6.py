"""The division by 6 (Markstein's correction step after a multiplication by
RN(1/6)) equals CUDA's correctly rounded __fdiv_rn(a, 6) for every binary32 a
in [0, 8], and the decode's branch-free E4M3 scale byte of a / 6 equals the
byte of that correctly rounded quotient: the check program compiles the
library's own device helpers and compares all 1,090,519,041 inputs on the
GPU."""
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "nvfp4_kv_cache_bd_gb300", "csrc")


def test_div6_matches_ieee_division_on_all_block_maxima():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "div6_check")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", CSRC,
                        os.path.join(HERE, "div6_check.cu"), "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    words = out.split()
    assert words[0] == "checked" and int(words[1]) == 0x41000001, out
    assert int(words[3]) == 0, out
    assert words[6:8] == ["scale", "mismatches"] and int(words[8]) == 0, out
