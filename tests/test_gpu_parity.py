"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Bars: packed K/V records and packed query bytes bit-exact (the fp32 q.mu
field within 1e-5 relative); attention outputs within max-abs 2e-3 and
relative-L2 1e-3 of the oracle's fp64 attention on the same quantized
operands.
"""
import numpy as np
import pytest
import torch

import nvfp4_kv_cache_bd_gb300 as bd
from nvfp4_kv_cache_bd_gb300 import synth
from tests import cases

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3


def same_output(x, y):
    """Two decode outputs of the same inputs: finite and bit for bit equal
    (every page goes to a fixed consumer warp, and warps and splits are
    merged in a fixed order)."""
    assert np.isfinite(x).all() and np.isfinite(y).all()
    assert np.array_equal(x, y), np.abs(x - y).max()


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    build.build_oracle()


def check(spec: cases.Spec, attn=True):
    c = cases.build(spec)
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c, pool_only=not attn)
    diff = np.nonzero(gpu["pool"] != ora["pool"])[0]
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"
    assert np.array_equal(cases.strip_qmu(c, gpu["qp"]), cases.strip_qmu(c, ora["qp"]))
    np.testing.assert_allclose(cases.qmu_of(c, gpu["qp"]), cases.qmu_of(c, ora["qp"]), rtol=1e-5, atol=1e-4)
    assert gpu["bf16_unchanged"]
    if attn:
        mx, rl = cases.attn_errors(gpu["out"], ora["out"])
        assert mx < MAX_ABS and rl < REL_L2, (mx, rl)
    assert bd.read_device_error(c.ctx) == bd.OK
    return c, gpu, ora


def test_single_sequence_4k_full_recipe():
    """One layer, 32 q / 8 kv heads, context 4096: 16 sink + 31 pages + 112 tail."""
    check(cases.Spec(lens=[4096], seed=0, tau=1.0))


def test_ragged_batch_edge_lengths():
    lens = [1, 5, 16, 17, 143, 144, 16 + 128 * 2 + 1, 16 + 128 * 3 + 127, 16 + 128 * 9]
    check(cases.Spec(lens=lens, seed=3))


@pytest.mark.parametrize("tau", [0.0, 0.5, 4.0, 448.0])
def test_tau_sweep(tau):
    check(cases.Spec(lens=[16 + 128 * 6 + 50, 900], seed=11, tau=tau))


@pytest.mark.parametrize("kw", [
    dict(p_mode=bd.P_AMAX6),
    dict(p_mode=bd.P_NONE),
    dict(p_c=1, tau=0.5),
    dict(rotation=0, centering=0, key_search=0, terms=1),
    dict(rotation=1, centering=0),
    dict(rotation=0, centering=1),
    dict(terms=1),
    dict(key_search=0),
])
def test_recipe_switches(kw):
    check(cases.Spec(lens=[16 + 128 * 5 + 77, 300], seed=21, **kw))


@pytest.mark.parametrize("kw", [dict(), dict(rotation=0, centering=0), dict(terms=1)])
def test_mxfp4(kw):
    check(cases.Spec(lens=[16 + 128 * 7 + 3, 16 + 128 * 2 + 100], seed=31, fmt=1, **kw))


def test_unshuffled_and_single_page():
    check(cases.Spec(lens=[16 + 128], seed=41, shuffle=False))


def test_writer_rounding_ties():
    """Values on every E2M1 tie and saturation point, with g = 1 and block
    amax 6 so that the E4M3 scale is exactly 1 and x * (1/S) = x."""
    spec = cases.Spec(lens=[16 + 128 * 2], seed=51, rotation=0, centering=0, key_search=0)
    c = cases.build(spec)
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.1, 0.3, 5.5, 4.5, 1.0, 0.0, 0.5, 2.0])
    vals = ties.repeat(8)
    sign = torch.where(torch.arange(128) % 3 == 0, -1.0, 1.0)
    row = (vals * sign)
    row[::16] = 6.0
    kp = row.repeat(c.k_pages.shape[0], 128, 8, 1).to(torch.bfloat16)
    kp[:, ::7, :, 13] = -0.0
    c.k_pages = kp.contiguous()
    c.v_pages = kp.flip(-1).contiguous()
    c.gk = c.gv = 1.0
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c, pool_only=True)
    assert np.array_equal(gpu["pool"], ora["pool"])


def test_writer_search_ties():
    """Key blocks whose {4,6} squared errors tie exactly in binary32 (the
    amax->6 scale is kept), and would flip to amax->4 if x - v*S were rounded
    once (tests/golden/tie_blocks.json): every key block of two pages is one
    of them, at every lane and token position."""
    import json
    import os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tie_blocks.json")))
    blocks = torch.tensor(fx["blocks_bf16"], dtype=torch.int32)                # [n][16]
    spec = cases.Spec(lens=[16 + 128 * 2], seed=52, rotation=0, centering=0, key_search=1)
    c = cases.build(spec)
    n_blk = c.k_pages.numel() // 16
    idx = (torch.arange(n_blk) * 7) % blocks.shape[0]
    kp = blocks[idx].to(torch.int16).view(torch.bfloat16).reshape(c.k_pages.shape)
    c.k_pages = kp.contiguous()
    c.gk = fx["g"]
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c, pool_only=True)
    assert np.array_equal(gpu["pool"], ora["pool"])


def test_writer_extreme_scales():
    """Tiny and huge per-tensor scales: E4M3 subnormal and saturated block scales."""
    for gk, gv in ((1e-4, 3e-5), (10.0, 50.0), (1e-30, 1e30)):
        c = cases.build(cases.Spec(lens=[16 + 128 * 3], seed=61))
        c.gk, c.gv = gk, gv
        gpu = cases.run_gpu(c)
        ora = cases.run_oracle(c, pool_only=True)
        assert np.array_equal(gpu["pool"], ora["pool"]), (gk, gv)


@pytest.mark.parametrize("fmt", [0, 1])
def test_writer_zero_blocks_and_extreme_magnitudes(fmt):
    """Raw values reach the quantizer (no centering / rotation): zero blocks,
    bf16 subnormals (MX exponent clamps at -127) and values near the bf16
    maximum (the larger MX candidate overflows and loses the search)."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 2], seed=71, fmt=fmt, rotation=0, centering=0))
    kp, vp = c.k_pages.clone(), c.v_pages.clone()
    for t in (kp, vp):
        t[0, :, :, :32] = 0.0
        t[0, 5, 3, 32:64] = 1e-39
        t[0, 6, 1, 64:96] = -3e-40
        t[1, 9, 2, :] = 3e38
        t[1, 10, 4, 96:] = -2.5e38
    c.k_pages, c.v_pages = kp, vp
    c.gk = c.gv = 1.0
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c, pool_only=True)
    assert np.array_equal(gpu["pool"], ora["pool"])


@pytest.mark.parametrize("fmt", [0, 1])
def test_writer_large_rotated_keys(fmt):
    """Large keys whose Hadamard sums stay finite (128 * 1e36 < fp32 max)."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 2], seed=72, fmt=fmt))
    kp = c.k_pages.clone()
    kp[1, 9, 2, :] = 1e36
    kp[1, 11, 5, ::3] = -7e35
    c.k_pages = kp
    c.gk = 1e30   # the largest per-tensor scale the API accepts; blocks saturate at 448
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c, pool_only=True)
    assert np.array_equal(gpu["pool"], ora["pool"])


def test_bounded_wait_reports_timeout():
    ctx = bd.Context(bd.make_config())
    assert bd.read_device_error(ctx) == bd.OK
    bd.selftest_bounded_wait(ctx, 20000)
    assert bd.read_device_error(ctx) == bd.ERR_TIMEOUT
    assert bd.read_device_error(ctx) == bd.OK     # reading resets the word
    ctx.close()


def test_identical_calls_are_bitwise_equal():
    """The writer, the query quantizer and the decode are bitwise
    deterministic: page 4 r + w of a split goes to consumer warp w, a CTA
    merges its warps in order, and the last split to finish merges all splits
    in split order."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 40 + 9], seed=81))
    a = cases.run_gpu(c)
    b = cases.run_gpu(c)
    assert np.array_equal(a["pool"], b["pool"]) and np.array_equal(a["qp"], b["qp"])
    same_output(a["out"], b["out"])


def test_empty_splits_ignore_workspace_garbage():
    """A batch whose short sequence leaves splits without pages, on a first
    call into a workspace full of NaN: the empty splits' unwritten O must not
    reach the output (the same result as with a zeroed workspace)."""
    c = cases.build(cases.Spec(lens=[700, 16 + 128 * 9 + 3], seed=77))
    gpu = cases.run_gpu(c)   # zeroed workspace
    ora = cases.run_oracle(c)
    mx, rl = cases.attn_errors(gpu["out"], ora["out"])
    assert mx < MAX_ABS and rl < REL_L2
    dev = "cuda"
    bt = torch.from_numpy(c.block_table).to(dev)
    B = bt.shape[0]
    ws = torch.full((bd.decode_workspace_size(c.ctx, B, bt.shape[1]) // 4 + 1,), float("nan"),
                    dtype=torch.float32, device=dev)
    out = torch.full((B, 32, 128), float("nan"), device=dev)
    bd.decode_attention(c.ctx, 0, torch.from_numpy(gpu["qp"]).to(dev), c.q.to(dev), torch.from_numpy(gpu["pool"]).to(dev),
                        bt, torch.from_numpy(c.seq_lens).to(dev), *[x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k,
                                                                                          c.tail_v)],
                        c.spec.tau, c.gk, c.gv, out, ws)
    torch.cuda.synchronize()
    same_output(out.cpu().double().numpy(), gpu["out"])


def test_workspace_needs_no_initialization_and_is_reusable():
    """The workspace holds only split partials, each written before it is
    read: one workspace that starts as garbage serves many calls, layers and
    batch shapes."""
    ctx = bd.Context(bd.make_config(num_layers=2))
    shapes = ([16 + 128 * 20 + 5], [700, 16 + 128 * 9], [16 + 128 * 20 + 5])
    # the size depends on the call's shape (its split layout), not only on B:
    # one workspace shared by several shapes is sized for the largest need
    ws = None
    for rep, lens in enumerate(shapes):
        c = cases.build(cases.Spec(lens=lens, seed=90 + rep), ctx=ctx)
        if ws is None:
            need = max(bd.decode_workspace_size(ctx, len(ls), max([1] + [synth.split_tokens(L)[1] for L in ls]))
                       for ls in shapes)
            ws = torch.full((need // 4 + 1,), float("nan"), dtype=torch.float32, device="cuda")
        gpu = cases.run_gpu(c)
        ora = cases.run_oracle(c)
        mx, rl = cases.attn_errors(gpu["out"], ora["out"])
        assert mx < MAX_ABS and rl < REL_L2
        # the same inputs again through one shared workspace, three times
        B = len(lens)
        dev = "cuda"
        pool = torch.from_numpy(gpu["pool"]).to(dev)
        qp = torch.from_numpy(gpu["qp"]).to(dev)
        q = c.q.to(dev)
        bt = torch.from_numpy(c.block_table).to(dev)
        sl = torch.from_numpy(c.seq_lens).to(dev)
        args = [x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k, c.tail_v)]
        ws_need = bd.decode_workspace_size(ctx, B, bt.shape[1])
        assert ws_need <= ws.numel() * 4
        for _ in range(3):
            out = torch.full((B, 32, 128), float("nan"), device=dev)
            bd.decode_attention(ctx, 0, qp, q, pool, bt, sl, *args, c.spec.tau, c.gk, c.gv, out, ws)
            torch.cuda.synchronize()
            same_output(out.cpu().double().numpy(), gpu["out"])
    assert bd.read_device_error(ctx) == bd.OK


@pytest.mark.parametrize("tau", [0.0, 4.0, 448.0])
def test_two_level_pages_use_each_pages_own_max(tau):
    """The probability quantizer's reference maximum is each page's own
    (reading A7): two FP4 pages whose keys are constant at two levels (page 1
    holds half of page 0's key row; the sink holds page 0's row), values +1.5
    and -1.5 on the pages and 0 in the sink.  The CPU pins show that the
    oracle's output here is the per-page closed form and that a maximum over
    both pages would miss it by more than five times this tolerance."""
    c = cases.build(cases.Spec(lens=[16 + 2 * 128], seed=52, tau=tau))
    kA = c.sink_k[0, 0].clone()
    kB = (kA.float() * 0.5).to(torch.bfloat16)
    c.sink_k[0] = kA
    c.sink_v.zero_()
    c.k_pages = torch.stack([kA.expand(128, 8, 128), kB.expand(128, 8, 128)]).contiguous()
    vp = torch.empty(2, 128, 8, 128, dtype=torch.bfloat16)
    vp[0], vp[1] = 1.5, -1.5
    c.v_pages = vp
    c.gv = 0.25
    gpu = cases.run_gpu(c)
    ora = cases.run_oracle(c)
    assert np.array_equal(gpu["pool"], ora["pool"])
    mx, rl = cases.attn_errors(gpu["out"], ora["out"])
    assert mx < MAX_ABS and rl < REL_L2, (mx, rl)
    assert bd.read_device_error(c.ctx) == bd.OK


def test_out_of_range_pages_are_skipped_and_reported():
    """Device-resident indexes outside the declared pool (bd_config.pool_pages)
    are never dereferenced: the writer skips such a destination, the decode
    leaves such a page out, and both record BD_ERR_INVALID_ARG.  The pool
    handed to the library sits two pages into a larger allocation, so pages
    -2, -1, n and n + 1 are still inside it and nothing could fault even if a
    check were missing; the bytes there must keep their fill value."""
    n = 5
    spec = cases.Spec(lens=[16 + 128 * n + 40, 16 + 128 * 2 + 9], seed=93, shuffle=False, spare_pages=0)
    c0 = cases.build(spec)
    npages = c0.nphys
    spec.pool_pages = npages
    c = cases.build(spec)
    dev = "cuda"
    H, rec = 8, c.rec
    page_bytes = H * 2 * rec
    big = torch.full(((npages + 4) * page_bytes,), cases.FILL, dtype=torch.uint8, device=dev)
    pool = big[2 * page_bytes:(npages + 2) * page_bytes]
    bd.set_key_shift(c.ctx, 0, c.mu)
    kp = torch.cat([c.k_pages, c.k_pages[:1]]).to(dev)
    vp = torch.cat([c.v_pages, c.v_pages[:1]]).to(dev)
    dst = torch.from_numpy(np.concatenate([c.dst, [npages]]).astype(np.int32)).to(dev)
    bd.quantize_kv_pages(c.ctx, 0, kp, vp, dst, c.gk, c.gv, pool)
    torch.cuda.synchronize()
    assert bd.read_device_error(c.ctx) == bd.ERR_INVALID_ARG
    ora = cases.run_oracle(c, pool_only=True)
    assert np.array_equal(pool.cpu().numpy(), ora["pool"])
    outside = torch.cat([big[:2 * page_bytes], big[(npages + 2) * page_bytes:]])
    assert bool((outside == cases.FILL).all())
    # decode with entries n (one past the pool) and -1 in the block table
    c.block_table[0, 1] = npages
    c.block_table[0, 3] = -1
    c.block_table[1, 0] = npages + 1
    B = len(spec.lens)
    q = c.q.to(dev)
    qp = torch.zeros(B, c.qstride, dtype=torch.uint8, device=dev)
    bd.quantize_query(c.ctx, 0, q, qp)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    args = [x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k, c.tail_v)]
    out = torch.full((B, 32, 128), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(bd.decode_workspace_size(c.ctx, B, bt.shape[1]) // 4 + 1, dtype=torch.float32, device=dev)
    bd.decode_attention(c.ctx, 0, qp, q, pool, bt, sl, *args, c.spec.tau, c.gk, c.gv, out, ws)
    torch.cuda.synchronize()
    assert bd.read_device_error(c.ctx) == bd.ERR_INVALID_ARG
    ref = cases.run_oracle(c)["out"]
    mx, rl = cases.attn_errors(out.cpu().double().numpy(), ref)
    assert mx < MAX_ABS and rl < REL_L2, (mx, rl)


def test_negative_and_overlong_lengths():
    """A negative length counts as 0 (zero output) and a length past the
    block table's capacity keeps its first max_blocks pages; both are
    reported in the device error word."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 3 + 50, 16 + 128 * 3 + 50], seed=94))
    gpu = cases.run_gpu(c)
    assert bd.read_device_error(c.ctx) == bd.OK
    dev = "cuda"
    B = 2
    sl = torch.tensor([-3, 16 + 128 * 7 + 50], dtype=torch.int32, device=dev)   # capacity: 3 pages + 127
    out = torch.full((B, 32, 128), float("nan"), dtype=torch.float32, device=dev)
    bt = torch.from_numpy(c.block_table).to(dev)
    ws = torch.zeros(bd.decode_workspace_size(c.ctx, B, bt.shape[1]) // 4 + 1, dtype=torch.float32, device=dev)
    bd.decode_attention(c.ctx, 0, torch.from_numpy(gpu["qp"]).to(dev), c.q.to(dev),
                        torch.from_numpy(gpu["pool"]).to(dev), bt, sl,
                        *[x.to(dev) for x in (c.sink_k, c.sink_v, c.tail_k, c.tail_v)], c.spec.tau, c.gk, c.gv,
                        out, ws)
    torch.cuda.synchronize()
    assert bd.read_device_error(c.ctx) == bd.ERR_INVALID_ARG
    c.seq_lens = sl.cpu().numpy()
    ref = cases.run_oracle(c)["out"]
    o = out.cpu().double().numpy()
    assert not o[0].any()
    mx, rl = cases.attn_errors(o, ref)
    assert mx < MAX_ABS and rl < REL_L2, (mx, rl)


@pytest.mark.parametrize("fmt,rotation,centering,terms", [(0, 1, 1, 2), (1, 1, 1, 2), (0, 0, 0, 1), (1, 1, 0, 1),
                                                          (0, 1, 1, 1)])
def test_fused_query_matches_the_two_calls(fmt, rotation, centering, terms):
    """bd_decode_attention without a packed query quantizes the query inside
    the decode with the same code and order as bd_quantize_query, so the
    output is bit-identical to quantize_query followed by the decode; it also
    meets the oracle's tolerance."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 7 + 5, 300, 16 + 128 * 12], seed=140 + fmt + 2 * terms, fmt=fmt,
                               rotation=rotation, centering=centering, terms=terms))
    two = cases.run_gpu(c)
    one = cases.run_gpu(c, fused_query=True)
    assert np.array_equal(one["out"], two["out"]), np.nanmax(np.abs(one["out"] - two["out"]))
    ora = cases.run_oracle(c)
    mx, rl = cases.attn_errors(one["out"], ora["out"])
    assert mx < MAX_ABS and rl < REL_L2


@pytest.mark.parametrize("hkv", [1, 2, 4])
def test_fused_query_with_fewer_kv_heads(hkv):
    """With fewer kv heads the token has fewer query heads than the decode
    CTA has threads: the items past 4 * hkv heads compute on zeros, and the
    warp whose items are the CTA's own query heads (warp h) still covers
    them whole.  Fused output bit-identical to the two calls, and within
    the oracle's tolerance."""
    c = cases.build(cases.Spec(lens=[16 + 128 * 5 + 9, 16 + 128 * 2], seed=170 + hkv, hkv=hkv))
    two = cases.run_gpu(c)
    one = cases.run_gpu(c, fused_query=True)
    assert np.array_equal(one["out"], two["out"]), np.nanmax(np.abs(one["out"] - two["out"]))
    ora = cases.run_oracle(c)
    mx, rl = cases.attn_errors(one["out"], ora["out"])
    assert mx < MAX_ABS and rl < REL_L2


def test_fused_query_on_a_multi_wave_grid():
    """20 sequences x 8 kv heads x (1 + 1) splits exceed one wave of two CTAs
    per SM: without a packed query the call quantizes it with the query
    kernel into the workspace first.  Same bytes, same output."""
    c = cases.build(cases.Spec(lens=[16 + 128 * (1 + i % 3) + 7 * i for i in range(20)], seed=160))
    two = cases.run_gpu(c)
    one = cases.run_gpu(c, fused_query=True)
    assert np.array_equal(one["out"], two["out"]), np.nanmax(np.abs(one["out"] - two["out"]))
    ora = cases.run_oracle(c)
    mx, rl = cases.attn_errors(one["out"], ora["out"])
    assert mx < MAX_ABS and rl < REL_L2
