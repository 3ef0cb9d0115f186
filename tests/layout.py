"""Test-side reader of the packed byte layouts (written independently of the
oracle and of the CUDA path, from the layout the public header documents).

K record (per page, KV head): codes in groups of 8 tokens x 32 dims: the
byte of dims d, d+1 (even d in the low nibble) of token t is at
(t//8)*512 + (d//32)*128 + (t%8)*16 + (d%32)//2; then the scales: block b of
token t at 8192 + (b//4)*512 + (t%32)*16 + (t//32)*4 + b%4.
V record: codes[8 groups][8 pairs][8 slots][16 B]; the byte of head dim d
holds token 16i+2p (low nibble) and token 16i+2p+1 (high nibble) and sits at
slot (d // 16) ^ 2 (p % 4), byte d % 16; scales[8][8][nb][2] (token 16i+2p
first).
nb = 8 E4M3 bytes (NVFP4, 16-element blocks) or 4 UE8M0 bytes (MXFP4, 32).
Pool: records ordered [page][kv_head][K, V].
"""
from __future__ import annotations

import numpy as np

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def e4m3_table() -> np.ndarray:
    out = np.zeros(256, np.float64)
    for b in range(256):
        e, m = (b >> 3) & 15, b & 7
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        out[b] = -v if b & 0x80 else v
    out[0x7F] = out[0xFF] = np.nan
    return out


E4M3 = e4m3_table()


def nblocks(fmt: int) -> int:
    return 8 if fmt == 0 else 4


def record_bytes(fmt: int) -> int:
    return 8192 + 128 * nblocks(fmt)


def scale_values(fmt: int, sbytes: np.ndarray) -> np.ndarray:
    if fmt == 0:
        return E4M3[sbytes]
    return np.ldexp(1.0, sbytes.astype(np.int64) - 127)


def k_record(fmt: int, rec: np.ndarray):
    """-> (codes [128][128] uint8, scale bytes [128][nb], values [128][128] fp64 without g)."""
    nb = nblocks(fmt)
    # [t//8][d//32][t%8][(d%32)//2] -> [t][d//2]
    by = rec[:8192].reshape(16, 4, 8, 16).transpose(0, 2, 1, 3).reshape(128, 64)
    codes = np.empty((128, 128), np.uint8)
    codes[:, 0::2] = by & 0xF
    codes[:, 1::2] = by >> 4
    t = np.arange(128)[:, None]
    b = np.arange(nb)[None, :]
    sb = rec[8192 + (b // 4) * 512 + (t % 32) * 16 + (t // 32) * 4 + b % 4]
    vals = E2M1[codes] * np.repeat(scale_values(fmt, sb), 128 // nb, axis=1)
    return codes, sb, vals


def v_record(fmt: int, rec: np.ndarray):
    """Same as k_record for a V record (token order restored)."""
    nb = nblocks(fmt)
    raw = rec[:8192].reshape(8, 8, 8, 16)
    by = np.empty((8, 8, 128), np.uint8)
    for p in range(8):
        for c in range(8):
            by[:, p, 16 * c:16 * c + 16] = raw[:, p, c ^ (2 * (p % 4))]
    codes = np.empty((128, 128), np.uint8)
    sbr = rec[8192:8192 + 128 * nb].reshape(8, 8, nb, 2)
    sb = np.empty((128, nb), np.uint8)
    for i in range(8):
        for p in range(8):
            codes[16 * i + 2 * p] = by[i, p] & 0xF
            codes[16 * i + 2 * p + 1] = by[i, p] >> 4
            sb[16 * i + 2 * p] = sbr[i, p, :, 0]
            sb[16 * i + 2 * p + 1] = sbr[i, p, :, 1]
    vals = E2M1[codes] * np.repeat(scale_values(fmt, sb), 128 // nb, axis=1)
    return codes, sb, vals


def pool_record(pool: np.ndarray, fmt: int, num_kv_heads: int, page: int, head: int, kv: int) -> np.ndarray:
    rb = record_bytes(fmt)
    off = ((page * num_kv_heads + head) * 2 + kv) * rb
    return pool[off:off + rb]


def qpack_stride(num_q_heads: int) -> int:
    raw = num_q_heads * (2 * 64 + 2 * 8 + 4) + 16
    return (raw + 255) // 256 * 256


def query_record(fmt: int, num_q_heads: int, rec: np.ndarray):
    """-> (Qhat [Hq][128] fp64 summed over terms incl. g, g[2], qmu[Hq], codes [2][Hq][128], scale bytes)."""
    Hq, nb = num_q_heads, nblocks(fmt)
    cb = rec[:2 * Hq * 64].reshape(2, Hq, 64)
    codes = np.empty((2, Hq, 128), np.uint8)
    codes[..., 0::2] = cb & 0xF
    codes[..., 1::2] = cb >> 4
    so = 2 * Hq * 64
    sb = rec[so:so + 2 * Hq * nb].reshape(2, Hq, nb)
    go = so + 2 * Hq * 8
    g = rec[go:go + 8].view(np.float32).copy()
    qmu = rec[go + 16:go + 16 + 4 * Hq].view(np.float32).copy()
    vals = E2M1[codes] * np.repeat(scale_values(fmt, sb), 128 // nb, axis=2)
    if fmt == 0:
        vals = vals * g.astype(np.float64)[:, None, None]
    return vals.sum(0), g, qmu, codes, sb
