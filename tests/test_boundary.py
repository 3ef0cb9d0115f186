"""Host-side tests of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU."""
import ctypes
import math
import os
import re

import pytest

import nvfp4_kv_cache_bd_gb300 as bd
from nvfp4_kv_cache_bd_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bd.h")


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return bd.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_exports(L):
    decl = declared_functions()
    assert decl == sorted(bd.EXPORTS)
    for name in decl:
        assert hasattr(L, name), name


def test_exported_symbols_via_nm(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (bd_\w+)", out))
    assert set(declared_functions()) <= exported


def test_status_strings(L):
    for code, text in [(0, "ok"), (-1, "invalid argument"), (-2, "unsupported"), (-4, "workspace"),
                       (-5, "timed out")]:
        assert text in bd.status_string(code)


def cfg(**kw):
    return bd.make_config(**kw)


@pytest.mark.parametrize("kw,status", [
    (dict(p_c=4), bd.ERR_INVALID_ARG),          # the probability kernel supports c = 1 or c = 8
    (dict(p_c=0), bd.ERR_INVALID_ARG),
    (dict(query_terms=3), bd.ERR_INVALID_ARG),
    (dict(p_mode=7), bd.ERR_INVALID_ARG),
    (dict(format=2), bd.ERR_INVALID_ARG),
    (dict(rotation=2), bd.ERR_INVALID_ARG),
    (dict(num_layers=0), bd.ERR_INVALID_ARG),
    (dict(pool_pages=-1), bd.ERR_INVALID_ARG),
    (dict(head_dim=64), bd.ERR_UNSUPPORTED),
    (dict(page_size=16), bd.ERR_UNSUPPORTED),
    (dict(sink_tokens=4), bd.ERR_UNSUPPORTED),
    (dict(num_q_heads=16), bd.ERR_UNSUPPORTED),
    (dict(num_kv_heads=32, num_q_heads=128), bd.ERR_UNSUPPORTED),
])
def test_create_rejects(L, kw, status):
    with pytest.raises(bd.BDError) as e:
        bd.Context(cfg(**kw))
    assert e.value.status == status


def test_create_accepts_recipe_variants(L):
    for kw in (dict(), dict(format=1), dict(p_c=1), dict(p_mode=bd.P_AMAX6), dict(p_mode=bd.P_NONE),
               dict(rotation=0, centering=0, key_search=0, query_terms=1), dict(num_kv_heads=1, num_q_heads=4)):
        ctx = bd.Context(cfg(**kw))
        assert ctx.record_bytes == (9216 if kw.get("format", 0) == 0 else 8704)
        assert ctx.query_packed_bytes % 256 == 0
        ctx.close()


def test_null_and_range_arguments(L):
    ctx = bd.Context(cfg(num_layers=2))
    h = ctx.handle
    P = ctypes.c_void_p
    fake = P(0x10000)
    s = P(0)
    # writer: null pointers, n < 0, bad layer, bad g
    assert L.bd_quantize_kv_pages(h, 0, None, fake, fake, 1, 1.0, 1.0, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_kv_pages(h, 0, fake, fake, fake, -1, 1.0, 1.0, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_kv_pages(h, 2, fake, fake, fake, 1, 1.0, 1.0, fake, s) == bd.ERR_INVALID_ARG
    for gk in (0.0, -1.0, math.nan, math.inf, 1e-35):
        assert L.bd_quantize_kv_pages(h, 0, fake, fake, fake, 1, gk, 1.0, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_kv_pages(h, 0, P(0x10008), fake, fake, 1, 1.0, 1.0, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_kv_pages(h, 0, None, None, None, 0, 1.0, 1.0, None, s) == bd.OK    # n = 0: no-op
    # query
    assert L.bd_quantize_query(h, 0, None, 1, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_query(h, 0, fake, -2, fake, s) == bd.ERR_INVALID_ARG
    assert L.bd_quantize_query(h, 0, None, 0, None, s) == bd.OK
    # append: null pointers, bad layer, unaligned buffers, bad g; B = 0 is a no-op
    app = [h, 0, fake, fake, fake, fake, 4, fake, fake, fake, fake, 2, 1.0, 1.0, fake, s]
    for i in (2, 3, 4, 7, 8, 9, 10):
        bad = list(app)
        bad[i] = None
        assert L.bd_append_kv(*bad) == bd.ERR_INVALID_ARG
    bad = list(app)
    bad[1] = 2
    assert L.bd_append_kv(*bad) == bd.ERR_INVALID_ARG
    bad = list(app)
    bad[9] = P(0x10008)
    assert L.bd_append_kv(*bad) == bd.ERR_INVALID_ARG
    bad = list(app)
    bad[12] = math.nan
    assert L.bd_append_kv(*bad) == bd.ERR_INVALID_ARG
    bad = list(app)
    bad[5] = None   # block_table missing while max_blocks > 0
    assert L.bd_append_kv(*bad) == bd.ERR_INVALID_ARG
    bad = list(app)
    bad[11] = 0
    assert L.bd_append_kv(*bad) == bd.OK
    # decode: tau must be finite and in [0, 448]
    ws_need = L.bd_decode_workspace_size(h, 1, 4)
    assert ws_need > 0
    args = lambda tau, ws_bytes=ws_need, gk=1.0: (h, 0, fake, fake, fake, fake, 4, fake, fake, fake, fake, fake, 1,
                                                  tau, gk, 1.0, fake, fake, ws_bytes, s)
    for tau in (-0.5, 448.5, math.nan, math.inf):
        assert L.bd_decode_attention(*args(tau)) == bd.ERR_INVALID_ARG
    assert L.bd_decode_attention(*args(1.0, gk=math.nan)) == bd.ERR_INVALID_ARG
    assert L.bd_decode_attention(*args(1.0, ws_bytes=ws_need - 1)) == bd.ERR_WORKSPACE
    bad = list(args(1.0))
    bad[3] = None  # q (raw query)
    assert L.bd_decode_attention(*bad) == bd.ERR_INVALID_ARG
    # no packed query: the decode quantizes q itself (checks pass; with no
    # GPU here the launch then fails), for up to 32 query heads
    bad = list(args(1.0))
    bad[2] = None
    assert L.bd_decode_attention(*bad) != bd.ERR_INVALID_ARG
    wide = bd.Context(bd.make_config(num_layers=1, num_q_heads=64, num_kv_heads=16))
    assert wide.cfg.num_q_heads == 64
    wargs = list(args(1.0, ws_bytes=L.bd_decode_workspace_size(wide.handle, 1, 4)))
    wargs[0] = wide.handle
    wargs[2] = None
    assert L.bd_decode_attention(*wargs) == bd.ERR_UNSUPPORTED
    wide.close()
    assert L.bd_set_key_shift(h, 5, fake) == bd.ERR_INVALID_ARG
    assert L.bd_selftest_bounded_wait(h, 0, s) == bd.ERR_INVALID_ARG
    assert L.bd_read_device_error(h, s, None) == bd.ERR_INVALID_ARG
    # copy: nothing to do, null, unaligned and overlapping ranges are settled
    # before any CUDA call; a pointer CUDA does not know is refused after its
    # attribute query (here: no GPU, so the query itself fails)
    assert L.bd_copy_async(None, None, 0, s) == bd.OK
    assert L.bd_copy_async(None, fake, 16, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(fake, None, 16, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(0x10008), P(0x20000), 16, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(0x10000), P(0x10010), 32, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(0x10000), P(0x20000), 64, s) in (bd.ERR_INVALID_ARG, bd.ERR_CUDA)
    ctx.close()


def test_workspace_size_monotone(L):
    ctx = bd.Context(cfg())
    sizes = [bd.decode_workspace_size(ctx, B, mb) for B, mb in ((1, 1), (1, 1023), (4, 1023), (32, 512))]
    assert all(s > 0 for s in sizes)
    assert bd.decode_workspace_size(ctx, 0, 10) == 0
    ctx.close()


def test_key_shift_rejects_non_finite(L):
    import torch
    ctx = bd.Context(cfg())
    mu = torch.zeros(8, 128)
    mu[3, 5] = float("nan")
    with pytest.raises(bd.BDError):
        bd.set_key_shift(ctx, 0, mu)
    ctx.close()
