"""Reconstruction-error and ablation report, and tau / c sensitivity, on
seeded synthetic data (no model or dataset needed).

For each quantization scheme the library's GPU path packs the pages, packs
the query and runs the decode; this module then measures, on the host:

- the relative RMS error of the dequantized keys and values against the
  bf16 inputs (keys compared in the original domain: rotation undone,
  key mean added back), over the FP4 pages;
- the attention output's relative L2 and max-abs error against exact fp64
  softmax attention over the same bf16 inputs (sink and tail included).

The schemes switch the recipe's parts one at a time (BitDecoding-FP4
evaluation config, RECIPE: key smoothing, Hadamard rotation, adaptive {4,6}
key scales, two query terms; probability_environment: the probability
quantizer's mode, c and tau; KV_MODES: NVFP4 vs MXFP4 scales).  The
sensitivity sweep varies tau and c of the amax2-or-amax6 probability mode.

    python -m nvfp4_kv_cache_bd_gb300.ablation [--ctx 16384] [--batch 4] [--json out.json]
"""
from __future__ import annotations

import argparse
import json
import math

import numpy as np
import torch

import nvfp4_kv_cache_bd_gb300 as bd
from nvfp4_kv_cache_bd_gb300 import synth

H, HQ, D = 8, 32, 128

BASE = dict(format=bd.FORMAT_NVFP4, key_search=1, rotation=1, centering=1, query_terms=2,
            p_mode=bd.P_AMAX2_OR_AMAX6, p_c=8)
SCHEMES = [
    ("full recipe", {}),
    ("no Hadamard rotation", dict(rotation=0)),
    ("no key centering", dict(centering=0)),
    ("no rotation, no centering", dict(rotation=0, centering=0)),
    ("amax6-only key scales", dict(key_search=0)),
    ("one query term", dict(query_terms=1)),
    ("probabilities not quantized", dict(p_mode=bd.P_NONE)),
    ("probabilities amax6, c = 1", dict(p_mode=bd.P_AMAX6, p_c=1)),
    ("MXFP4 scales", dict(format=bd.FORMAT_MXFP4)),
]

# ------------------------------------------------------- host dequantizer --
# Byte layouts of include/bd.h: a K record is codes in groups of 8 tokens x
# 32 dims (the byte of dims d, d+1 of token t at (t/8)*512 + (d/32)*128 +
# (t%8)*16 + (d%32)/2, even d in the low nibble) then nb/4 scale-factor
# groups of 512 B (block b of token t at 8192 + (b/4)*512 + (t%32)*16 +
# (t/32)*4 + b%4); a V record is codes[8][8][128 B] where the byte of head
# dim d in row (i, p) holds token 16i+2p (low nibble) and token 16i+2p+1
# (high nibble) and sits at 16-byte slot (d // 16) ^ 2 (p % 4), then
# scales[8][8][nb][2].  nb = 8 E4M3 bytes (NVFP4) or 4 UE8M0 bytes (MXFP4).
# A packed query (stride S) holds codes[2 terms][Hq][64 B] (K's nibble
# order), scales[2][Hq][nb], then g1, g2 and q.mu[Hq] as float32.

_E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, 0, -.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def _e4m3_values() -> np.ndarray:
    b = np.arange(256)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.where(b & 0x80, -v, v)


_E4M3 = _e4m3_values()


def _scale(fmt, sb):
    return _E4M3[sb] if fmt == bd.FORMAT_NVFP4 else np.ldexp(1.0, sb.astype(np.int64) - 127)


def dequantize_pool(pool: np.ndarray, fmt: int, pages: np.ndarray, gk: float, gv: float):
    """-> (K, V) fp64 [n_pages][128 tok][H][128] of the given physical pages,
    in the stored domain (keys still rotated and centered), per-tensor
    scales applied (NVFP4)."""
    nb = 8 if fmt == bd.FORMAT_NVFP4 else 4
    rb = 8192 + 128 * nb
    recs = pool.reshape(-1, H, 2, rb)[pages]                       # [n][H][2][rb]
    # K codes in groups of 8 tokens x 32 dims: [t//8][d//32][t%8][(d%32)//2] -> [t][d//2]
    kc = recs[:, :, 0, :8192].reshape(-1, H, 16, 4, 8, 16).transpose(0, 1, 2, 4, 3, 5).reshape(-1, H, 128, 64)
    kcodes = np.stack([kc & 0xF, kc >> 4], axis=-1).reshape(-1, H, 128, 128)
    # K scales: block b of token t at 8192 + (b//4)*512 + (t%32)*16 + (t//32)*4 + b%4
    t = np.arange(128)[:, None]
    b = np.arange(nb)[None, :]
    ks = recs[:, :, 0, 8192 + (b // 4) * 512 + (t % 32) * 16 + (t // 32) * 4 + b % 4]
    k = _E2M1[kcodes] * np.repeat(_scale(fmt, ks), 128 // nb, axis=-1)
    vslot = recs[:, :, 1, :8192].reshape(-1, H, 8, 8, 8, 16)
    p = np.arange(8)[:, None]
    vc = vslot[:, :, :, p, np.arange(8)[None, :] ^ (2 * (p % 4))].reshape(-1, H, 8, 8, 128)
    vcodes = np.stack([vc & 0xF, vc >> 4], axis=4).reshape(-1, H, 128, 128)   # tokens 16i + 2p + (0 | 1)
    vs = recs[:, :, 1, 8192:8192 + 128 * nb].reshape(-1, H, 8, 8, nb, 2)
    vs = np.stack([vs[..., 0], vs[..., 1]], axis=4).reshape(-1, H, 128, nb)
    v = _E2M1[vcodes] * np.repeat(_scale(fmt, vs), 128 // nb, axis=-1)
    if fmt == bd.FORMAT_NVFP4:
        k, v = k * gk, v * gv
    return k.transpose(0, 2, 1, 3), v.transpose(0, 2, 1, 3)


def dequantize_query(qp: np.ndarray, fmt: int, hq: int = HQ):
    """-> (Qhat [B][hq][128] fp64, the sum of both terms with their scales in
    the rotated domain, q.mu [B][hq]) from packed query records [B][S]."""
    nb = 8 if fmt == bd.FORMAT_NVFP4 else 4
    B = qp.shape[0]
    codes = qp[:, :2 * hq * 64].reshape(B, 2, hq, 64)
    c = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(B, 2, hq, 128)
    sb = qp[:, 2 * hq * 64:2 * hq * 64 + 2 * hq * nb].reshape(B, 2, hq, nb)
    goff = 2 * hq * 64 + 2 * hq * 8
    g = np.ascontiguousarray(qp[:, goff:goff + 8]).view(np.float32).astype(np.float64)      # [B][2]
    qmu = np.ascontiguousarray(qp[:, goff + 16:goff + 16 + 4 * hq]).view(np.float32).astype(np.float64)
    terms = _E2M1[c] * np.repeat(_scale(fmt, sb), 128 // nb, axis=-1)
    if fmt == bd.FORMAT_NVFP4:
        terms = terms * g[:, :, None, None]
    return terms.sum(axis=1), qmu


def _fwht_rows(x: np.ndarray) -> np.ndarray:
    """Normalized Sylvester Hadamard transform along the last axis (128)."""
    x = x.copy()
    h = 1
    while h < D:
        y = x.reshape(*x.shape[:-1], D // (2 * h), 2, h)
        a, b = y[..., 0, :].copy(), y[..., 1, :].copy()
        y[..., 0, :], y[..., 1, :] = a + b, a - b
        h *= 2
    return x / math.sqrt(D)


# ------------------------------------------------------------- reference --

def exact_attention(q, k, v):
    """fp64 softmax attention for one sequence: q [HQ][D], k/v [L][H][D]."""
    out = np.empty((HQ, D))
    for j in range(HQ):
        kh, vh = k[:, j // (HQ // H)], v[:, j // (HQ // H)]
        s = kh @ q[j] / math.sqrt(D)
        p = np.exp(s - s.max())
        out[j] = (p / p.sum()) @ vh
    return out


# ------------------------------------------------------------------ runs --

class Data:
    def __init__(self, ctx_len, batch, seed, dev):
        self.lens = [ctx_len] * batch
        self.mu, mask = synth.key_mean(H, seed, dev)
        self.kv = [synth.keys_values(ctx_len, H, 100 * seed + b, dev, mu=self.mu, mask=mask) for b in range(batch)]
        self.q = synth.query(batch, HQ, seed, dev)
        self.split = synth.split_tokens(ctx_len)


def run_scheme(data: Data, cfgkw: dict, taus=(1.0,), dev="cuda"):
    B = len(data.lens)
    ns, n, nt = data.split
    ctx = bd.Context(bd.make_config(**cfgkw))
    bd.set_key_shift(ctx, 0, data.mu)
    allk = torch.cat([k for k, _ in data.kv])
    allv = torch.cat([v for _, v in data.kv])
    gk, gv = synth.gscales(allk, allv, data.mu, bool(cfgkw["rotation"]), bool(cfgkw["centering"]))
    gk, gv = (gk or 1.0), (gv or 1.0)
    pool = torch.zeros(ctx.pool_bytes(B * n), dtype=torch.uint8, device=dev)
    bt = torch.arange(B * n, dtype=torch.int32, device=dev).view(B, n)
    kp = torch.cat([k[16:16 + 128 * n].view(n, 128, H, D) for k, _ in data.kv])
    vp = torch.cat([v[16:16 + 128 * n].view(n, 128, H, D) for _, v in data.kv])
    bd.quantize_kv_pages(ctx, 0, kp, vp, bt.reshape(-1), gk, gv, pool)
    qp = torch.zeros(B, ctx.query_packed_bytes, dtype=torch.uint8, device=dev)
    bd.quantize_query(ctx, 0, data.q, qp)
    sk = torch.stack([k[:16] for k, _ in data.kv])
    sv = torch.stack([v[:16] for _, v in data.kv])
    tk = torch.zeros(B, 128, H, D, dtype=torch.bfloat16, device=dev)
    tv = torch.zeros_like(tk)
    for b, (k, v) in enumerate(data.kv):
        tk[b, :nt], tv[b, :nt] = k[16 + 128 * n:], v[16 + 128 * n:]
    sl = torch.tensor(data.lens, dtype=torch.int32, device=dev)
    ws = torch.empty(bd.decode_workspace_size(ctx, B, n) // 4 + 1, dtype=torch.float32, device=dev)
    outs = {}
    for tau in taus:
        out = torch.empty(B, HQ, D, dtype=torch.float32, device=dev)
        bd.decode_attention(ctx, 0, qp, data.q, pool, bt, sl, sk, sv, tk, tv, tau, gk, gv, out, ws)
        outs[tau] = out.double().cpu().numpy()
    torch.cuda.synchronize()
    if bd.read_device_error(ctx) != bd.OK:
        raise RuntimeError("device error word set")
    return ctx, pool.cpu().numpy(), qp.cpu().numpy(), gk, gv, outs


def key_value_errors(data: Data, cfgkw: dict, pool: np.ndarray, gk: float, gv: float):
    B = len(data.lens)
    n = data.split[1]
    kh, vh = dequantize_pool(pool, cfgkw["format"], np.arange(B * n), gk, gv)
    kh = kh.reshape(B, n * 128, H, D)
    vh = vh.reshape(B, n * 128, H, D)
    mu = data.mu.double().cpu().numpy()
    if cfgkw["rotation"]:
        kh = _fwht_rows(kh)
    if cfgkw["centering"]:
        kh = kh + mu
    kref = np.stack([k[16:16 + 128 * n].double().cpu().numpy() for k, _ in data.kv])
    vref = np.stack([v[16:16 + 128 * n].double().cpu().numpy() for _, v in data.kv])
    rel = lambda a, r: float(np.linalg.norm(a - r) / np.linalg.norm(r))
    return rel(kh, kref), rel(vh, vref)


def error_budget(data: Data, cfgkw: dict, pool: np.ndarray, qp: np.ndarray, gk: float, gv: float,
                 out: np.ndarray, ref: np.ndarray) -> dict:
    """Where the attention error comes from, on the FP4 pages (the BF16 sink
    and tail are exact throughout), in fp64 on the host from the library's
    own bytes:

    - logits: the scores Qhat . Khat (+ q.mu with centering) against the
      exact q . k, and A1 = softmax attention with those scores, exact P and
      exact V, against the exact attention A0;
    - values: A2 = A1 with the dequantized V, against A1;
    - probabilities: the decode's output (FP4 P, f16 MMAs) against A2.
    Relative L2 norms; logit_rms in natural-log units (scores / sqrt(d))."""
    B = len(data.lens)
    n = data.split[1]
    fmt = cfgkw["format"]
    kh, vh = dequantize_pool(pool, fmt, np.arange(B * n), gk, gv)   # stored domain
    kh = kh.reshape(B, n * 128, H, D)
    vh = vh.reshape(B, n * 128, H, D)
    qh, qmu = dequantize_query(qp, fmt)
    fp = slice(16, 16 + 128 * n)
    a1 = np.empty_like(ref)
    a2 = np.empty_like(ref)
    ds2 = s2 = 0.0
    cnt = 0
    for b, (k, v) in enumerate(data.kv):
        k64, v64 = k.double().cpu().numpy(), v.double().cpu().numpy()
        q64 = data.q[b].double().cpu().numpy()
        for j in range(HQ):
            h = j // (HQ // H)
            s_ex = k64[:, h] @ q64[j] / math.sqrt(D)
            s_hat = s_ex.copy()
            s_hat[fp] = (kh[b, :, h] @ qh[b, j] + (qmu[b, j] if cfgkw["centering"] else 0.0)) / math.sqrt(D)
            d = s_hat[fp] - s_ex[fp]
            ds2 += float(d @ d)
            s2 += float(s_ex[fp] @ s_ex[fp])
            cnt += d.size
            p = np.exp(s_hat - s_hat.max())
            p /= p.sum()
            a1[b, j] = p @ v64[:, h]
            vq = v64[:, h].copy()
            vq[fp] = vh[b, :, h]
            a2[b, j] = p @ vq
    rel = lambda x, y: float(np.linalg.norm(x - y) / np.linalg.norm(y))
    return dict(logit_rms=math.sqrt(ds2 / max(cnt, 1)), logit_rel=math.sqrt(ds2 / max(s2, 1e-300)),
                logits_rel_l2=rel(a1, ref), values_rel_l2=rel(a2, a1), probabilities_rel_l2=rel(out, a2),
                total_rel_l2=rel(out, ref))


def attention_errors(data: Data, out: np.ndarray, ref: np.ndarray):
    d = out - ref
    return float(np.linalg.norm(d) / np.linalg.norm(ref)), float(np.max(np.abs(d)))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ctx", type=int, default=16384)
    ap.add_argument("--batch", type=int, default=4)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--json", default=None)
    args = ap.parse_args()
    dev = "cuda"
    data = Data(args.ctx, args.batch, args.seed, dev)
    q64 = data.q.double().cpu().numpy()
    ref = np.stack([exact_attention(q64[b], k.double().cpu().numpy(), v.double().cpu().numpy())
                    for b, (k, v) in enumerate(data.kv)])
    res = {"workload": f"{args.batch} sequences x {args.ctx} tokens, 32 q / 8 kv heads, d128, seed {args.seed}",
           "schemes": {}, "tau_sweep": {}}
    print(f"| scheme | K rel-RMSE | V rel-RMSE | attention rel-L2 | attention max-abs |")
    print(f"|---|---|---|---|---|")
    budgets = {}
    for name, over in SCHEMES:
        kw = dict(BASE, **over)
        ctx, pool, qp, gk, gv, outs = run_scheme(data, kw, dev=dev)
        ek, ev = key_value_errors(data, kw, pool, gk, gv)
        rl, mx = attention_errors(data, outs[1.0], ref)
        budgets[name] = error_budget(data, kw, pool, qp, gk, gv, outs[1.0], ref)
        res["schemes"][name] = dict(config=kw, k_rel_rmse=ek, v_rel_rmse=ev, attn_rel_l2=rl, attn_max_abs=mx,
                                    error_budget=budgets[name])
        print(f"| {name} | {ek:.4f} | {ev:.4f} | {rl:.5f} | {mx:.5f} |")
        ctx.close()
    print()
    print("| scheme | logit RMS | logit rel | attention from logits | + values | + probabilities | total |")
    print("|---|---|---|---|---|---|---|")
    for name, e in budgets.items():
        print(f"| {name} | {e['logit_rms']:.4f} | {e['logit_rel']:.4f} | {e['logits_rel_l2']:.4f} | "
              f"{e['values_rel_l2']:.4f} | {e['probabilities_rel_l2']:.4f} | {e['total_rel_l2']:.4f} |")
    print()
    print("| c | " + " | ".join(f"tau {t:g}" for t in (0, 0.25, 0.5, 1, 2, 4, 8, 448)) + " |")
    print("|---|" + "---|" * 8)
    taus = (0.0, 0.25, 0.5, 1.0, 2.0, 4.0, 8.0, 448.0)
    for c in (1, 8):
        kw = dict(BASE, p_c=c)
        ctx, _, _, _, _, outs = run_scheme(data, kw, taus=taus, dev=dev)
        row = {}
        for t in taus:
            rl, mx = attention_errors(data, outs[t], ref)
            row[str(t)] = dict(attn_rel_l2=rl, attn_max_abs=mx)
        res["tau_sweep"][f"c={c}"] = row
        print(f"| {c} | " + " | ".join(f"{row[str(t)]['attn_rel_l2']:.5f}" for t in taus) + " |")
        ctx.close()
    if args.json:
        with open(args.json, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()
