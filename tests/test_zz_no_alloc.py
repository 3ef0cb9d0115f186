"""bd_decode_attention_noalloc against bd_decode_attention, through the C ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc
(code running inside another framework's memory pool, a plugin handed only
its input and output buffers, a process whose GPU memory is reserved up
front).  Its split scratch is a fixed array inside the library that every
call reuses, so two calls in a row must both reproduce the workspace entry
point's output.
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


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    c = cases.build(cases.Spec(lens=[16 + 128 * 6 + 33, 700, 16 + 128 * 2], seed=123))
    ref = cases.run_gpu(c)      # writer + query + decode with a caller workspace
    dev = "cuda"
    B = len(c.spec.lens)
    pool = torch.from_numpy(ref["pool"]).to(dev)
    qp = torch.from_numpy(ref["qp"]).to(dev)
    q = c.q.to(dev)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    sk, sv, tk, tv = (x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k, c.tail_v))
    for _ in range(2):
        out = torch.full((B, 32, 128), float("nan"), dtype=torch.float32, device=dev)
        bd.decode_attention_noalloc(c.ctx, 0, qp, q, pool, bt, sl, sk, sv, tk, tv, c.spec.tau, c.gk, c.gv, out)
        torch.cuda.synchronize()
        mx, rl = cases.attn_errors(out.cpu().double().numpy(), ref["out"])
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
