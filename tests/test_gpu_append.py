"""bd_append_kv through the C ABI: tokens appended one decode step at a time
land in the BF16 sink and tail, the tail page a token completes is packed
into its pool slot bit for bit like the oracle's writer, and the decode over
the resulting cache matches the oracle over the same token stream."""
import numpy as np
import pytest
import torch

import nvfp4_kv_cache_bd_gb300 as bd
import oracle
from nvfp4_kv_cache_bd_gb300 import synth
from tests import cases

pytestmark = pytest.mark.gpu

H, HQ, D = 8, 32, 128
MAX_ABS, REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    build.build_oracle()


def u16(t):
    return t.detach().cpu().contiguous().view(torch.uint16).numpy()


class Cache:
    """One sequence's hybrid cache on the GPU, filled from a token stream."""

    def __init__(self, ctx, k, v, L0, block_row, nphys, gk, gv, dev="cuda"):
        self.ctx, self.gk, self.gv = ctx, gk, gv
        rec = ctx.record_bytes
        self.pool = torch.full((nphys * H * 2 * rec,), cases.FILL, dtype=torch.uint8, device=dev)
        self.bt = torch.tensor([block_row], dtype=torch.int32, device=dev)
        ns, n, nt = synth.split_tokens(L0)
        if n:
            bd.quantize_kv_pages(ctx, 0, k[16:16 + 128 * n].view(n, 128, H, D).to(dev),
                                 v[16:16 + 128 * n].view(n, 128, H, D).to(dev), self.bt[0, :n], gk, gv, self.pool)
        self.sk = torch.zeros(1, 16, H, D, dtype=torch.bfloat16, device=dev)
        self.sv = torch.zeros_like(self.sk)
        self.tk = torch.zeros(1, 128, H, D, dtype=torch.bfloat16, device=dev)
        self.tv = torch.zeros_like(self.tk)
        self.sk[0, :ns], self.sv[0, :ns] = k[:ns].to(dev), v[:ns].to(dev)
        self.tk[0, :nt], self.tv[0, :nt] = k[16 + 128 * n:L0].to(dev), v[16 + 128 * n:L0].to(dev)


def test_append_fills_the_completed_page_and_decode_matches():
    dev = "cuda"
    ctx = bd.Context(bd.make_config())
    L0, steps = 16 + 128 * 2 + 120, 20           # the 8th appended token completes page 2
    T = L0 + steps
    mu, mask = synth.key_mean(H, 31)
    k, v = synth.keys_values(T, H, 31, mu=mu, mask=mask)
    gk, gv = synth.gscales(k, v, mu, True, True)
    bd.set_key_shift(ctx, 0, mu)
    block_row = [5, 2, 7, 0]
    c = Cache(ctx, k, v, L0, block_row, 8, gk, gv)
    before = c.pool.cpu().numpy()
    sl = torch.zeros(1, dtype=torch.int32, device=dev)
    for t in range(steps):
        sl.fill_(L0 + t)
        bd.append_kv(ctx, 0, k[L0 + t].view(1, H, D).to(dev), v[L0 + t].view(1, H, D).to(dev), sl, c.bt,
                     c.sk, c.sv, c.tk, c.tv, gk, gv, c.pool)
    torch.cuda.synchronize()
    assert bd.read_device_error(ctx) == bd.OK
    pool = c.pool.cpu().numpy()

    # the oracle packs pages 0..2 (tokens 16..399) into physical pages 5, 2, 7
    ocfg = oracle.make_config()
    ref_pool = np.full_like(before, cases.FILL)
    oracle.quantize_kv_pages(ocfg, u16(k[16:16 + 384].view(3, 128, H, D)), u16(v[16:16 + 384].view(3, 128, H, D)),
                             np.array(block_row[:3], np.int32), mu.numpy(), gk, gv, ref_pool)
    assert np.array_equal(pool, ref_pool), "packed pool differs from the oracle writer"
    # the tail now holds tokens 400..411, the sink is untouched
    assert torch.equal(c.tk[0, :12].cpu(), k[400:412]) and torch.equal(c.tv[0, :12].cpu(), v[400:412])
    assert torch.equal(c.sk[0].cpu(), k[:16])

    # decode at length T over the appended cache against the oracle
    q = synth.query(1, HQ, 31)
    qp = torch.zeros(1, ctx.query_packed_bytes, dtype=torch.uint8, device=dev)
    bd.quantize_query(ctx, 0, q.to(dev), qp)
    out = torch.empty(1, HQ, D, dtype=torch.float32, device=dev)
    ws = torch.empty(bd.decode_workspace_size(ctx, 1, 4) // 4 + 1, dtype=torch.float32, device=dev)
    bd.decode_attention(ctx, 0, qp, q.to(dev), c.pool, c.bt, torch.tensor([T], dtype=torch.int32, device=dev),
                        c.sk, c.sv, c.tk, c.tv, 1.0, gk, gv, out, ws)
    torch.cuda.synchronize()
    tk = torch.zeros(1, 128, H, D, dtype=torch.bfloat16)
    tv = torch.zeros_like(tk)
    tk[0, :12], tv[0, :12] = k[400:412], v[400:412]
    oqp = oracle.quantize_query(ocfg, u16(q), mu.numpy())
    ref = oracle.decode_attention(ocfg, oqp, u16(q), mu.numpy(), ref_pool, np.array([block_row], np.int32),
                                  np.array([T], np.int32), u16(k[:16].view(1, 16, H, D)),
                                  u16(v[:16].view(1, 16, H, D)), u16(tk), u16(tv), 1.0, gk, gv)
    mx, rl = cases.attn_errors(out.cpu().double().numpy(), ref)
    assert mx < MAX_ABS and rl < REL_L2, (mx, rl)


def test_append_batch_in_sink_and_at_a_page_boundary():
    """Sequence 0 is still in its sink, sequence 1 completes its first page."""
    dev = "cuda"
    ctx = bd.Context(bd.make_config())
    mu, mask = synth.key_mean(H, 32)
    ks = [synth.keys_values(200, H, 40 + b, mu=mu, mask=mask) for b in range(2)]
    gk, gv = synth.gscales(torch.cat([x[0] for x in ks]), torch.cat([x[1] for x in ks]), mu, True, True)
    bd.set_key_shift(ctx, 0, mu)
    lens = [10, 16 + 127]
    pool = torch.full((4 * H * 2 * ctx.record_bytes,), cases.FILL, dtype=torch.uint8, device=dev)
    bt = torch.tensor([[1, 0], [3, 2]], dtype=torch.int32, device=dev)
    sk = torch.zeros(2, 16, H, D, dtype=torch.bfloat16, device=dev)
    sv, tk, tv = torch.zeros_like(sk), torch.zeros(2, 128, H, D, dtype=torch.bfloat16, device=dev), None
    tv = torch.zeros_like(tk)
    for b, L in enumerate(lens):
        k, v = ks[b]
        ns = min(L, 16)
        sk[b, :ns], sv[b, :ns] = k[:ns].to(dev), v[:ns].to(dev)
        if L > 16:
            tk[b, :L - 16], tv[b, :L - 16] = k[16:L].to(dev), v[16:L].to(dev)
    before = np.full(pool.numel(), cases.FILL, np.uint8)
    knew = torch.stack([ks[b][0][lens[b]] for b in range(2)]).to(dev)
    vnew = torch.stack([ks[b][1][lens[b]] for b in range(2)]).to(dev)
    bd.append_kv(ctx, 0, knew, vnew, torch.tensor(lens, dtype=torch.int32, device=dev), bt, sk, sv, tk, tv, gk, gv,
                 pool)
    torch.cuda.synchronize()
    assert bd.read_device_error(ctx) == bd.OK
    assert torch.equal(sk[0, 10].cpu(), ks[0][0][10]) and torch.equal(sv[0, 10].cpu(), ks[0][1][10])
    ref_pool = before.copy()
    oracle.quantize_kv_pages(oracle.make_config(), u16(ks[1][0][16:144].view(1, 128, H, D)),
                             u16(ks[1][1][16:144].view(1, 128, H, D)), np.array([3], np.int32), mu.numpy(), gk, gv,
                             ref_pool)
    assert np.array_equal(pool.cpu().numpy(), ref_pool)


def test_append_without_a_page_slot_records_an_error_and_writes_no_page():
    dev = "cuda"
    ctx = bd.Context(bd.make_config())
    pool = torch.full((2 * H * 2 * ctx.record_bytes,), cases.FILL, dtype=torch.uint8, device=dev)
    bt = torch.zeros(1, 1, dtype=torch.int32, device=dev)           # room for page 0 only
    sk = torch.zeros(1, 16, H, D, dtype=torch.bfloat16, device=dev)
    sv, tk = torch.zeros_like(sk), torch.zeros(1, 128, H, D, dtype=torch.bfloat16, device=dev)
    tv = torch.zeros_like(tk)
    new = torch.ones(1, H, D, dtype=torch.bfloat16, device=dev)
    L = torch.tensor([16 + 128 + 127], dtype=torch.int32, device=dev)   # would complete page 1
    bd.append_kv(ctx, 0, new, new, L, bt, sk, sv, tk, tv, 1.0, 1.0, pool)
    torch.cuda.synchronize()
    assert bd.read_device_error(ctx) == bd.ERR_INVALID_ARG
    assert bool((pool == cases.FILL).all())
    assert bool((tk[0, 127] == 1).all())     # the token itself is stored
