"""Parity at the benchmark's full sizes, in the launch configuration the
benchmark times (the library picks the same splits for the same shapes).

- Single sequence at 32768 and 131072 tokens of context, layers 0, 17 and 35
  of the 36-layer workload (per-layer seed = layer): every packed byte the
  writer produces, the packed query, and the attention output of every head
  against the oracle; at 131072 tokens also the tau sweep {0, 0.5, 4, 448}.
- Batched decode: 32 sequences with lengths log-uniform in [1024, 65536],
  pages of all sequences interleaved in one pool, NVFP4 and MXFP4, each with
  rotation and centering on and off: every writer byte and every
  sequence's attention output.

The oracle work is spread over CPU processes (tests/fullsize.py).
"""
import numpy as np
import pytest
import torch

import nvfp4_kv_cache_bd_gb300 as bd
import oracle
from nvfp4_kv_cache_bd_gb300 import synth
from tests import cases
from tests.fullsize import OraclePool

pytestmark = pytest.mark.gpu

H, HQ, D = 8, 32, 128
MAX_ABS, REL_L2 = 2e-3, 1e-3
QMU_REL = 1e-5


@pytest.fixture(scope="module")
def opool():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    build.build_oracle()
    p = OraclePool()
    yield p
    p.close()


def u16(t):
    return t.detach().cpu().contiguous().view(torch.uint16).numpy()


def _qp_check(gpu_qp, ora_qp):
    off = 2 * HQ * 64 + 2 * HQ * 8 + 16
    a, b = gpu_qp.copy(), ora_qp.copy()
    qa = np.ascontiguousarray(a[:, off:off + 4 * HQ]).view(np.float32)
    qb = np.ascontiguousarray(b[:, off:off + 4 * HQ]).view(np.float32)
    a[:, off:off + 4 * HQ] = 0
    b[:, off:off + 4 * HQ] = 0
    assert np.array_equal(a, b), "packed query bytes differ"
    assert np.allclose(qa, qb, rtol=QMU_REL, atol=QMU_REL * max(1.0, float(np.max(np.abs(qb)))))


def _run_layer(opool, ctx, kw, layer, ctx_len, taus=(1.0,)):
    """One layer of the single-sequence workload through the GPU and the oracle."""
    dev = "cuda"
    mu, mask = synth.key_mean(H, layer, dev)
    k, v = synth.keys_values(ctx_len, H, layer, dev, mu=mu, mask=mask)
    gk, gv = synth.gscales(k, v, mu, bool(kw["rotation"]), bool(kw["centering"]))
    q = synth.query(1, HQ, layer, dev)
    n_sink, npages, n_tail = synth.split_tokens(ctx_len)
    bt = synth.page_permutation(npages, 0, dev).view(1, -1).contiguous()
    bd.set_key_shift(ctx, layer, mu)
    rec = ctx.record_bytes
    pool = torch.full((npages * H * 2 * rec,), cases.FILL, dtype=torch.uint8, device=dev)
    kp = k[16:16 + 128 * npages].view(npages, 128, H, D)
    vp = v[16:16 + 128 * npages].view(npages, 128, H, D)
    bd.quantize_kv_pages(ctx, layer, kp, vp, bt[0], gk, gv, pool)
    qp = torch.zeros(1, ctx.query_packed_bytes, dtype=torch.uint8, device=dev)
    bd.quantize_query(ctx, layer, q, qp)
    sk = torch.zeros(1, 16, H, D, dtype=torch.bfloat16, device=dev)
    sv = torch.zeros_like(sk)
    sk[0, :n_sink], sv[0, :n_sink] = k[:n_sink], v[:n_sink]
    tk = torch.zeros(1, 128, H, D, dtype=torch.bfloat16, device=dev)
    tv = torch.zeros_like(tk)
    tk[0, :n_tail], tv[0, :n_tail] = k[16 + 128 * npages:], v[16 + 128 * npages:]
    sl = torch.tensor([ctx_len], dtype=torch.int32, device=dev)
    ws = torch.empty(bd.decode_workspace_size(ctx, 1, npages) // 4 + 1, dtype=torch.float32, device=dev)
    outs = {}
    for tau in taus:
        out = torch.full((1, HQ, D), float("nan"), dtype=torch.float32, device=dev)
        bd.decode_attention(ctx, layer, qp, q, pool, bt, sl, sk, sv, tk, tv, tau, gk, gv, out, ws)
        outs[tau] = out
    torch.cuda.synchronize()
    assert bd.read_device_error(ctx) == bd.OK

    # the oracle on the same bf16 tensors
    ocfg = oracle.make_config(**kw)
    mu_np = mu.cpu().numpy()
    ora_pool = np.full(npages * H * 2 * rec, cases.FILL, np.uint8)
    opool.quantize_pages(kw, u16(kp), u16(vp), bt[0].cpu().numpy(), mu_np, gk, gv, ora_pool)
    assert np.array_equal(pool.cpu().numpy(), ora_pool), f"layer {layer}: packed pool differs"
    ora_qp = oracle.quantize_query(ocfg, u16(q), mu_np)
    _qp_check(qp.cpu().numpy(), ora_qp)
    for tau, out in outs.items():
        ref = oracle.decode_attention(ocfg, ora_qp, u16(q), mu_np, ora_pool, bt.cpu().numpy(),
                                      np.array([ctx_len], np.int32), u16(sk), u16(sv), u16(tk), u16(tv), tau, gk, gv)
        mx, rl = cases.attn_errors(out.cpu().double().numpy(), ref)
        assert mx < MAX_ABS and rl < REL_L2, (layer, tau, mx, rl)


FULL = dict(fmt=0, key_search=1, rotation=1, centering=1, query_terms=2, p_mode=2, p_c=8)


@pytest.mark.parametrize("ctx_len", [32768, 131072])
def test_single_sequence_layers_0_17_35(opool, ctx_len):
    ctx = bd.Context(bd.make_config(num_layers=36))
    for layer in (0, 17, 35):
        taus = (1.0, 0.0, 0.5, 4.0, 448.0) if (ctx_len == 131072 and layer == 0) else (1.0,)
        _run_layer(opool, ctx, FULL, layer, ctx_len, taus)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("recipe", [1, 0])
def test_batched_32_sequences(opool, fmt, recipe):
    """32 sequences, log-uniform lengths in [1024, 65536], their pages taken
    round-robin from one shared pool."""
    dev = "cuda"
    kw = dict(fmt=fmt, key_search=1, rotation=recipe, centering=recipe, query_terms=2, p_mode=2, p_c=8)
    ctx = bd.Context(bd.make_config(format=fmt, rotation=recipe, centering=recipe))
    lens = synth.log_uniform_lengths(32, 1024, 65536, 0)
    B = len(lens)
    splits = [synth.split_tokens(L) for L in lens]
    npg = [s[1] for s in splits]
    maxb = max(npg)
    # round-robin page allocation: physical page ids handed out one per
    # sequence in turn, so neighbouring pages belong to different sequences
    bt = np.zeros((B, maxb), np.int32)
    nxt, rnd = 0, 0
    while rnd < maxb:
        for b in range(B):
            if rnd < npg[b]:
                bt[b, rnd] = nxt
                nxt += 1
        rnd += 1
    total = nxt
    mu, mask = synth.key_mean(H, 4000, dev)
    bd.set_key_shift(ctx, 0, mu)
    seqs = [synth.keys_values(L, H, 4000 + b, dev, mu=mu, mask=mask) for b, L in enumerate(lens)]
    allk = torch.cat([s[0] for s in seqs])
    allv = torch.cat([s[1] for s in seqs])
    gk, gv = synth.gscales(allk, allv, mu, bool(recipe), bool(recipe))
    del allk, allv
    kpages = torch.cat([s[0][16:16 + 128 * n].view(n, 128, H, D) for s, n in zip(seqs, npg)])
    vpages = torch.cat([s[1][16:16 + 128 * n].view(n, 128, H, D) for s, n in zip(seqs, npg)])
    dst = np.concatenate([bt[b, :npg[b]] for b in range(B)]).astype(np.int32)
    rec = ctx.record_bytes
    pool = torch.full((total * H * 2 * rec,), cases.FILL, dtype=torch.uint8, device=dev)
    bd.quantize_kv_pages(ctx, 0, kpages, vpages, torch.from_numpy(dst).to(dev), gk, gv, pool)
    q = synth.query(B, HQ, 4000, dev)
    qp = torch.zeros(B, ctx.query_packed_bytes, dtype=torch.uint8, device=dev)
    bd.quantize_query(ctx, 0, q, qp)
    sk = torch.zeros(B, 16, H, D, dtype=torch.bfloat16, device=dev)
    sv = torch.zeros_like(sk)
    tk = torch.zeros(B, 128, H, D, dtype=torch.bfloat16, device=dev)
    tv = torch.zeros_like(tk)
    for b, ((ns, n, nt), (k, v)) in enumerate(zip(splits, seqs)):
        sk[b, :ns], sv[b, :ns] = k[:ns], v[:ns]
        tk[b, :nt], tv[b, :nt] = k[16 + 128 * n:], v[16 + 128 * n:]
    btd = torch.from_numpy(bt).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    ws = torch.empty(bd.decode_workspace_size(ctx, B, maxb) // 4 + 1, dtype=torch.float32, device=dev)
    out = torch.full((B, HQ, D), float("nan"), dtype=torch.float32, device=dev)
    bd.decode_attention(ctx, 0, qp, q, pool, btd, sl, sk, sv, tk, tv, 1.0, gk, gv, out, ws)
    torch.cuda.synchronize()
    assert bd.read_device_error(ctx) == bd.OK

    ocfg = oracle.make_config(**kw)
    mu_np = mu.cpu().numpy()
    ora_pool = np.full(total * H * 2 * rec, cases.FILL, np.uint8)
    opool.quantize_pages(kw, u16(kpages), u16(vpages), dst, mu_np, gk, gv, ora_pool)
    assert np.array_equal(pool.cpu().numpy(), ora_pool), "packed pool differs"
    ora_qp = oracle.quantize_query(ocfg, u16(q), mu_np)
    _qp_check(qp.cpu().numpy(), ora_qp)
    ref = opool.decode(kw, ora_qp, u16(q), mu_np, ora_pool, bt, np.array(lens, np.int32), u16(sk), u16(sv), u16(tk),
                       u16(tv), 1.0, gk, gv)
    mx, rl = cases.attn_errors(out.cpu().double().numpy(), ref)
    assert mx < MAX_ABS and rl < REL_L2, (fmt, recipe, mx, rl)
