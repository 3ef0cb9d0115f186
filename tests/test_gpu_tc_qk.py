"""The decode's tensor-core QK product (block-scaled tcgen05 MMA, FP4 x FP4
with E4M3 or UE8M0 block scales) on one page, against fp64 dot products of
the same dequantized operands.

The check program (tests/tc_qk_check.cu) runs the library's own device
helpers on a K record written by the library's page writer and a query
packed by its query quantizer; the expected scores come from the test-side
layout reader (tests/layout.py), which decodes the bytes independently of
both the CUDA path and the oracle.  A page whose keys live in one 16-dim
block has every score exact in fp32 (each is one block-scale product times a
sum of at most 12-bit integers), so those must match bit for bit; full pages
are held to the fp32 accumulation bound."""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from tests import cases, layout

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "nvfp4_kv_cache_bd_gb300", "csrc")


@pytest.fixture(scope="module")
def checker():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    build.build_oracle()
    d = tempfile.mkdtemp()
    exe = os.path.join(d, "tc_qk_check")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-I", CSRC,
                    os.path.join(HERE, "tc_qk_check.cu"), "-o", exe], check=True, capture_output=True)
    return exe


def run_check(exe, fmt, h, rec, qp):
    with tempfile.TemporaryDirectory() as d:
        fin, fout = os.path.join(d, "in.bin"), os.path.join(d, "out.bin")
        with open(fin, "wb") as f:
            f.write(np.array([fmt, h], np.int32).tobytes())
            f.write(np.ascontiguousarray(rec).tobytes())
            f.write(np.ascontiguousarray(qp).tobytes())
        r = subprocess.run([exe, fin, fout], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
        return np.fromfile(fout, np.float32).reshape(128, 8)


def expected(fmt, h, rec, qp):
    """fp64 scores [128][8] (column 2 hh + term) and the sum of |products|."""
    kvals = layout.k_record(fmt, rec)[2]                       # codes x block scales, no per-tensor scale
    _, _, _, qcodes, qsb = layout.query_record(fmt, 32, qp)
    nb = layout.nblocks(fmt)
    qvals = layout.E2M1[qcodes] * np.repeat(layout.scale_values(fmt, qsb), 128 // nb, axis=2)   # [2][32][128]
    rows = np.stack([qvals[term, 4 * h + hh] for hh in range(4) for term in range(2)])          # [8][128]
    return kvals @ rows.T, np.abs(kvals) @ np.abs(rows).T


def page_case(fmt, seed, one_block=False):
    c = cases.build(cases.Spec(lens=[16 + 128 + 3], seed=seed, fmt=fmt, rotation=0 if one_block else 1,
                               centering=0 if one_block else 1))
    if one_block:
        kp = c.k_pages.clone()
        kp[..., 16:] = 0.0
        c.k_pages = kp
    return c, cases.run_gpu(c)


@pytest.mark.parametrize("fmt", [0, 1])
def test_qk_page_one_block_is_exact(checker, fmt):
    c, gpu = page_case(fmt, 301, one_block=True)
    for h in (0, 3, 7):
        rec = layout.pool_record(gpu["pool"], fmt, 8, c.block_table[0, 0], h, 0)
        out = run_check(checker, fmt, h, rec, gpu["qp"][0])
        ref, _ = expected(fmt, h, rec, gpu["qp"][0])
        assert np.array_equal(out, ref.astype(np.float32)), np.abs(out - ref).max()


@pytest.mark.parametrize("fmt", [0, 1])
def test_qk_page_full_recipe(checker, fmt):
    c, gpu = page_case(fmt, 302)
    for h in range(8):
        rec = layout.pool_record(gpu["pool"], fmt, 8, c.block_table[0, 0], h, 0)
        out = run_check(checker, fmt, h, rec, gpu["qp"][0])
        ref, mag = expected(fmt, h, rec, gpu["qp"][0])
        # fp32 accumulation of 128 exact products: within a few ulps of the magnitude sum
        assert np.all(np.abs(out - ref) <= 2.0 ** -21 * mag + 1e-30), np.abs(out - ref).max()
