"""Seeded hybrid-cache test cases run through both the CUDA path (C ABI via
the package binding) and the CPU oracle, from the same synthetic inputs."""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np
import torch

import nvfp4_kv_cache_bd_gb300 as bd
import oracle
from nvfp4_kv_cache_bd_gb300 import synth

H, HQ, D = 8, 32, 128
FILL = 0xA5   # pool bytes outside the written records must keep this value


@dataclasses.dataclass
class Spec:
    lens: List[int]
    seed: int = 0
    fmt: int = 0
    rotation: int = 1
    centering: int = 1
    key_search: int = 1
    terms: int = 2
    p_mode: int = 2
    p_c: int = 8
    tau: float = 1.0
    shuffle: bool = True
    spare_pages: int = 2
    pool_pages: int = 0    # declared pool size (0: not declared)
    hkv: int = H           # kv heads (query heads: 4 per kv head)


class Case:
    pass


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint16).numpy()


def build(spec: Spec, ctx=None) -> Case:
    c = Case()
    c.spec = spec
    H, HQ = spec.hkv, 4 * spec.hkv
    B = len(spec.lens)
    mu, mask = synth.key_mean(H, spec.seed)
    c.mu = mu
    c.q = synth.query(B, HQ, spec.seed)
    splits = [synth.split_tokens(L) for L in spec.lens]
    npg = [s[1] for s in splits]
    total = sum(npg)
    nphys = total + spec.spare_pages
    perm = synth.page_permutation(nphys, spec.seed).numpy() if spec.shuffle else np.arange(nphys, dtype=np.int32)
    maxb = max([1] + npg)
    c.block_table = np.zeros((B, maxb), np.int32)
    c.sink_k = torch.zeros(B, 16, H, D, dtype=torch.bfloat16)
    c.sink_v = torch.zeros_like(c.sink_k)
    c.tail_k = torch.zeros(B, 128, H, D, dtype=torch.bfloat16)
    c.tail_v = torch.zeros_like(c.tail_k)
    kp, vp, dst, ks, vs = [], [], [], [], []
    off = 0
    for b, L in enumerate(spec.lens):
        k, v = synth.keys_values(L, H, spec.seed * 1000 + b, mu=mu, mask=mask)
        ks.append(k)
        vs.append(v)
        ns, n, nt = splits[b]
        c.sink_k[b, :ns] = k[:ns]
        c.sink_v[b, :ns] = v[:ns]
        c.tail_k[b, :nt] = k[16 + 128 * n:]
        c.tail_v[b, :nt] = v[16 + 128 * n:]
        if n:
            kp.append(k[16:16 + 128 * n].reshape(n, 128, H, D))
            vp.append(v[16:16 + 128 * n].reshape(n, 128, H, D))
            c.block_table[b, :n] = perm[off:off + n]
            dst.append(perm[off:off + n])
            off += n
    c.k_seqs, c.v_seqs = ks, vs
    c.k_pages = torch.cat(kp) if kp else torch.zeros(0, 128, H, D, dtype=torch.bfloat16)
    c.v_pages = torch.cat(vp) if vp else torch.zeros(0, 128, H, D, dtype=torch.bfloat16)
    c.dst = np.concatenate(dst).astype(np.int32) if dst else np.zeros(0, np.int32)
    c.seq_lens = np.array(spec.lens, np.int32)
    allk = torch.cat(ks) if sum(spec.lens) else torch.zeros(1, H, D, dtype=torch.bfloat16)
    allv = torch.cat(vs) if sum(spec.lens) else torch.zeros(1, H, D, dtype=torch.bfloat16)
    c.gk, c.gv = synth.gscales(allk, allv, mu, bool(spec.rotation), bool(spec.centering))
    if c.gk == 0.0:
        c.gk = 1.0
    if c.gv == 0.0:
        c.gv = 1.0
    c.nphys = nphys
    c.ocfg = oracle.make_config(num_q_heads=HQ, num_kv_heads=H, fmt=spec.fmt, key_search=spec.key_search,
                                rotation=spec.rotation,
                                centering=spec.centering, query_terms=spec.terms, p_mode=spec.p_mode, p_c=spec.p_c,
                                pool_pages=spec.pool_pages)
    c.ctx = ctx if ctx is not None else bd.Context(bd.make_config(
        num_q_heads=HQ, num_kv_heads=H, format=spec.fmt, key_search=spec.key_search, rotation=spec.rotation,
        centering=spec.centering,
        query_terms=spec.terms, p_mode=spec.p_mode, p_c=spec.p_c, pool_pages=spec.pool_pages))
    c.rec = oracle.record_bytes(c.ocfg)
    c.qstride = oracle.qpack_stride(c.ocfg)
    return c


def strip_qmu(c: Case, qp: np.ndarray) -> np.ndarray:
    """Packed query bytes with the fp32 q.mu field zeroed (it is compared with a tolerance)."""
    HQ = 4 * c.spec.hkv
    qp = qp.copy()
    off = 2 * HQ * 64 + 2 * HQ * 8 + 16
    qp[:, off:off + 4 * HQ] = 0
    return qp


def qmu_of(c: Case, qp: np.ndarray) -> np.ndarray:
    HQ = 4 * c.spec.hkv
    off = 2 * HQ * 64 + 2 * HQ * 8 + 16
    return np.ascontiguousarray(qp[:, off:off + 4 * HQ]).view(np.float32)


def run_gpu(c: Case, dev="cuda", stream=None, pool=None, fused_query=False) -> dict:
    """The library path: writer, query quantizer, decode.  fused_query: the
    decode takes no packed query and quantizes q itself (the packed query is
    still produced, for the fields compared elsewhere)."""
    B = len(c.spec.lens)
    H, HQ = c.spec.hkv, 4 * c.spec.hkv
    bd.set_key_shift(c.ctx, 0, c.mu)
    g = lambda t: t.to(dev)
    if pool is None:
        pool = torch.full((c.nphys * H * 2 * c.rec,), FILL, dtype=torch.uint8, device=dev)
    kp, vp = g(c.k_pages), g(c.v_pages)
    dst = torch.from_numpy(c.dst).to(dev)
    bd.quantize_kv_pages(c.ctx, 0, kp, vp, dst, c.gk, c.gv, pool, stream)
    q = g(c.q)
    qp = torch.zeros(B, c.qstride, dtype=torch.uint8, device=dev)
    bd.quantize_query(c.ctx, 0, q, qp, stream)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    sk, sv, tk, tv = g(c.sink_k), g(c.sink_v), g(c.tail_k), g(c.tail_v)
    out = torch.full((B, HQ, D), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(1, bd.decode_workspace_size(c.ctx, B, bt.shape[1])) // 4 + 1, dtype=torch.float32,
                     device=dev)
    bd.decode_attention(c.ctx, 0, None if fused_query else qp, q, pool, bt, sl, sk, sv, tk, tv, c.spec.tau, c.gk,
                        c.gv, out, ws, stream)
    torch.cuda.synchronize()
    res = dict(pool=pool.cpu().numpy(), qp=qp.cpu().numpy(), out=out.cpu().double().numpy())
    res["bf16_unchanged"] = all(torch.equal(a.cpu(), b) for a, b in
                                ((sk, c.sink_k), (sv, c.sink_v), (tk, c.tail_k), (tv, c.tail_v), (kp, c.k_pages),
                                 (vp, c.v_pages), (q, c.q)))
    return res


def run_oracle(c: Case, pool_only: bool = False) -> dict:
    H = c.spec.hkv
    pool = np.full(c.nphys * H * 2 * c.rec, FILL, np.uint8)
    if len(c.dst):
        oracle.quantize_kv_pages(c.ocfg, u16(c.k_pages), u16(c.v_pages), c.dst, c.mu.numpy(), c.gk, c.gv, pool)
    qp = oracle.quantize_query(c.ocfg, u16(c.q), c.mu.numpy())
    res = dict(pool=pool, qp=qp)
    if not pool_only:
        res["out"] = oracle.decode_attention(c.ocfg, qp, u16(c.q), c.mu.numpy(), pool, c.block_table, c.seq_lens,
                                             u16(c.sink_k), u16(c.sink_v), u16(c.tail_k), u16(c.tail_v),
                                             c.spec.tau, c.gk, c.gv)
    return res


def attn_errors(gpu_out: np.ndarray, ref: np.ndarray):
    """(max-abs, relative L2) of the attention output."""
    d = gpu_out - ref
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
