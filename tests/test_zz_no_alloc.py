"""bd_decode_attention_noalloc against bd_decode_attention, through the C ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc
(code running inside another framework's memory pool, a plugin handed only
its input and output buffers, a process whose GPU memory is reserved up
front).  Its split scratch is a fixed array inside the library that every
call reuses, so calls that follow an earlier call with another split layout
must still reproduce the workspace entry point's output.
"""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_bd_gb300 as bd
from tests import cases

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    build.build_oracle()


def _noalloc(c, pool, qp, out, dev="cuda"):
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    sk, sv, tk, tv = (x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k, c.tail_v))
    bd.decode_attention_noalloc(c.ctx, 0, qp, c.q.to(dev), pool, bt, sl, sk, sv, tk, tv, c.spec.tau, c.gk, c.gv,
                                out)
    torch.cuda.synchronize()


def test_noalloc_matches_workspace_entry_point_after_a_larger_call():
    """A larger call first (8 sequences of 40 pages: a different split layout
    over more of the shared array) whose values are NaN, so every partial O it
    leaves behind is NaN with a finite maximum and denominator.  Then a
    3-sequence call, twice: both must match the workspace entry point, which
    they cannot if any partial left over from an earlier call is read."""
    dev = "cuda"
    big = cases.build(cases.Spec(lens=[16 + 128 * 40 + 7] * 8, seed=124))
    ref_big = cases.run_gpu(big)
    pool = ref_big["pool"].copy().reshape(big.nphys, 8, 2, big.rec)
    pool[:, :, 1, 8192:] = 0x7F            # every V block scale is the E4M3 NaN
    big.sink_v = torch.full_like(big.sink_v, float("nan"))
    out = torch.zeros((8, 32, 128), dtype=torch.float32, device=dev)
    _noalloc(big, torch.from_numpy(pool.reshape(-1)).to(dev), torch.from_numpy(ref_big["qp"]).to(dev), out)
    assert bool(torch.isnan(out).all())

    c = cases.build(cases.Spec(lens=[16 + 128 * 6 + 33, 700, 16 + 128 * 2], seed=123), ctx=big.ctx)
    ref = cases.run_gpu(c)      # writer + query + decode with a caller workspace
    assert bd.decode_workspace_size(c.ctx, 3, c.block_table.shape[1]) != \
        bd.decode_workspace_size(c.ctx, 8, big.block_table.shape[1])
    pool = torch.from_numpy(ref["pool"]).to(dev)
    qp = torch.from_numpy(ref["qp"]).to(dev)
    ora = cases.run_oracle(c)   # the CPU oracle on the same packed pages and query
    for _ in range(2):
        out = torch.full((3, 32, 128), float("nan"), dtype=torch.float32, device=dev)
        _noalloc(c, pool, qp, out)
        got = out.cpu().double().numpy()
        # the same kernel and split layout as the workspace entry point: the same bits
        assert np.array_equal(got, ref["out"]), float(np.nanmax(np.abs(got - ref["out"])))
        mx, rl = cases.attn_errors(got, ora["out"])
        assert mx < MAX_ABS and rl < REL_L2, (mx, rl)
    assert bd.read_device_error(c.ctx) == bd.OK


def test_noalloc_rejects_calls_beyond_its_scratch():
    ctx = bd.Context(bd.make_config())
    fake = ctypes.c_void_p(0x10000)
    big_b = 4096
    assert bd.decode_workspace_size(ctx, big_b, 8) > (4 << 20)
    st = bd.lib().bd_decode_attention_noalloc(ctx.handle, 0, fake, fake, fake, fake, 8, fake, fake, fake, fake, fake,
                                              big_b, 1.0, 1.0, 1.0, fake, ctypes.c_void_p(0))
    assert st == bd.ERR_WORKSPACE
    ctx.close()
