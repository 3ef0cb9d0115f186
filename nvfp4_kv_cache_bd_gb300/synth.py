"""Seeded synthetic inputs shaped like the long-context decode workload.

This module only draws random tensors and picks per-tensor scales from
simple statistics; it holds none of the quantizer or attention arithmetic, so
the CUDA path and the CPU oracle can both be fed from it.

Recipe (Qwen3-4B-like heads: 32 query / 8 KV heads, head_dim 128):
  * Q, V ~ N(0, 1), rounded to bf16.
  * key mean mu[h, d] ~ N(0, std 2) per (layer, KV head, channel); 4 channels
    per (layer, KV head), chosen without replacement, are outliers: their
    mean and their noise are multiplied by 20.  K = noise + mu, rounded to
    bf16.  The key shift handed to the library is that generating mean.
  * per-tensor scales: g_V = max|V| / 2688 and, for K, the transformed key's
    bound / 2688 where the bound is max|K - mu| without rotation and
    max_t ||K_t - mu||_2 with rotation (an orthonormal rotation never moves a
    coordinate above the vector's 2-norm), so no E4M3 block scale saturates.
    2688 = 6 * 448 maps the bound onto the largest E2M1 value times the
    largest E4M3 scale.
"""
from __future__ import annotations

import math

import torch

D = 128
PAGE = 128
SINK = 16


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def key_mean(num_kv_heads: int, seed: int, device="cpu", n_outliers: int = 4):
    """mu [Hkv][D] fp32 and the outlier mask [Hkv][D] (bool)."""
    g = _gen(seed * 7919 + 1, device)
    mu = torch.randn(num_kv_heads, D, generator=g, device=device) * 2.0
    mask = torch.zeros(num_kv_heads, D, dtype=torch.bool, device=device)
    for h in range(num_kv_heads):
        idx = torch.randperm(D, generator=g, device=device)[:n_outliers]
        mask[h, idx] = True
    mu = torch.where(mask, mu * 20.0, mu)
    return mu, mask


def keys_values(num_tokens: int, num_kv_heads: int, seed: int, device="cpu", mu=None, mask=None):
    """K, V bf16 [T][Hkv][D] following the recipe above (mu/mask from key_mean)."""
    if mu is None:
        mu, mask = key_mean(num_kv_heads, seed, device)
    g = _gen(seed * 7919 + 2, device)
    noise = torch.randn(num_tokens, num_kv_heads, D, generator=g, device=device)
    noise = torch.where(mask.unsqueeze(0), noise * 20.0, noise)
    k = (noise + mu.unsqueeze(0)).to(torch.bfloat16)
    v = torch.randn(num_tokens, num_kv_heads, D, generator=g, device=device).to(torch.bfloat16)
    return k, v


def query(batch: int, num_q_heads: int, seed: int, device="cpu"):
    g = _gen(seed * 7919 + 3, device)
    return torch.randn(batch, num_q_heads, D, generator=g, device=device).to(torch.bfloat16)


def gscales(k, v, mu, rotation: bool, centering: bool):
    """(g_K, g_V) as python floats (binary32 values)."""
    kf = k.float()
    if centering:
        kf = kf - mu.to(kf.device).unsqueeze(0)
    if rotation:
        bound = kf.norm(dim=-1).max()
    else:
        bound = kf.abs().max()
    gk = torch.tensor(float(bound) / 2688.0, dtype=torch.float32).item()
    gv = torch.tensor(float(v.float().abs().max()) / 2688.0, dtype=torch.float32).item()
    return gk, gv


def page_permutation(n: int, seed: int, device="cpu"):
    """A seeded shuffle of physical page ids 0..n-1 (int32)."""
    g = _gen(seed * 7919 + 4, device)
    return torch.randperm(n, generator=g, device=device).to(torch.int32)


def log_uniform_lengths(batch: int, lo: int, hi: int, seed: int):
    """Sequence lengths round(exp(U[ln lo, ln hi])) (python ints)."""
    g = _gen(seed * 7919 + 5, "cpu")
    u = torch.rand(batch, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def split_tokens(L: int, sink: int = SINK, page: int = PAGE):
    """(n_sink, n_pages, n_tail) of a sequence of length L in the hybrid cache."""
    n_sink = min(L, sink)
    rest = max(0, L - sink)
    n_pages = rest // page
    return n_sink, n_pages, rest - n_pages * page
