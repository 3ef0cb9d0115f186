"""CPU oracle for the NVFP4 KV-cache hot path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``bd_oracle.c`` (plain C,
binary32 quantizer steps with round-to-nearest-even and no fused multiply-add,
binary64 attention) through ctypes and shares no code with the CUDA path.

Every function takes and returns numpy arrays; bf16 tensors travel as
``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile bd_oracle.c into liboracle.so next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


FMT_NVFP4, FMT_MXFP4 = 0, 1
P_NONE, P_AMAX6, P_AMAX2_OR_AMAX6 = 0, 1, 2
FLAG_QUANT_DENOM = 1


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "page_size", "sink_tokens", "format",
        "key_search", "rotation", "centering", "query_terms", "p_mode", "p_c", "pool_pages")]


def make_config(num_q_heads=32, num_kv_heads=8, fmt=FMT_NVFP4, key_search=1, rotation=1,
                centering=1, query_terms=2, p_mode=P_AMAX2_OR_AMAX6, p_c=8, sink_tokens=16,
                pool_pages=0) -> Config:
    return Config(num_q_heads, num_kv_heads, 128, 128, sink_tokens, fmt, key_search, rotation,
                  centering, query_terms, p_mode, p_c, pool_pages)


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        CP = ctypes.POINTER(Config)
        sig = {
            "or_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "or_e2m1_value": (ctypes.c_float, [ctypes.c_uint8]),
            "or_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "or_e4m3_value": (ctypes.c_float, [ctypes.c_uint8]),
            "or_e2m1_encode_n": (None, [P, P, I64]),
            "or_e4m3_encode_n": (None, [P, P, I64]),
            "or_block_sse": (ctypes.c_float, [P, P, ctypes.c_int]),
            "or_nvfp4_block": (None, [P, ctypes.c_int, ctypes.c_float, P, P, P]),
            "or_four_six_block": (ctypes.c_int, [P, ctypes.c_float, P, P, P, P, P]),
            "or_mx_block": (ctypes.c_int, [P, P, P, P, P, P]),
            "or_fwht128": (None, [P]),
            "or_rotate128": (None, [P]),
            "or_record_bytes": (I64, [CP]),
            "or_qpack_stride": (I64, [CP]),
            "or_mem_ratio": (ctypes.c_double, [CP]),
            "or_quantize_kv_pages": (ctypes.c_int, [CP, P, P, P, ctypes.c_int, P, ctypes.c_float,
                                                    ctypes.c_float, P]),
            "or_quantize_query": (ctypes.c_int, [CP, P, ctypes.c_int, P, P]),
            "or_decode_attention": (ctypes.c_int, [CP, P, P, P, P, P, ctypes.c_int, P, P, P, P, P,
                                                   ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_float, ctypes.c_int, P]),
            "or_attention_identity_quant": (ctypes.c_int, [CP, P, P, P, ctypes.c_int, P, P]),
            "or_p_block": (None, [P, ctypes.c_int, ctypes.c_int, ctypes.c_float, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---- scalar formats --------------------------------------------------------

def e2m1_encode(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint8)
    lib().or_e2m1_encode_n(_p(x), _p(out), x.size)
    return out


def e2m1_value(codes) -> np.ndarray:
    return np.array([lib().or_e2m1_value(int(c)) for c in np.asarray(codes).ravel()], np.float32)


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint8)
    lib().or_e4m3_encode_n(_p(x), _p(out), x.size)
    return out


def e4m3_value(b) -> np.ndarray:
    return np.array([lib().or_e4m3_value(int(c)) for c in np.asarray(b).ravel()], np.float32)


# ---- block quantizers ------------------------------------------------------

def nvfp4_block(x, m: int, g: float):
    x = _c(x, np.float32)
    codes = np.empty(16, np.uint8)
    sb = np.empty(1, np.uint8)
    xh = np.empty(16, np.float32)
    lib().or_nvfp4_block(_p(x), m, g, _p(codes), _p(sb), _p(xh))
    return codes, int(sb[0]), xh


def four_six_block(x, g: float):
    x = _c(x, np.float32)
    codes = np.empty(16, np.uint8)
    sb = np.empty(1, np.uint8)
    xh = np.empty(16, np.float32)
    e4 = np.empty(1, np.float32)
    e6 = np.empty(1, np.float32)
    m = lib().or_four_six_block(_p(x), g, _p(codes), _p(sb), _p(xh), _p(e4), _p(e6))
    return m, codes, int(sb[0]), xh, float(e4[0]), float(e6[0])


def mx_block(x):
    x = _c(x, np.float32)
    codes = np.empty(32, np.uint8)
    sb = np.empty(1, np.uint8)
    xh = np.empty(32, np.float32)
    ea = np.empty(1, np.float32)
    eb = np.empty(1, np.float32)
    e = lib().or_mx_block(_p(x), _p(codes), _p(sb), _p(xh), _p(ea), _p(eb))
    return e, codes, int(sb[0]), xh, float(ea[0]), float(eb[0])


def p_block(ptil, p_mode: int, p_c: int, tau: float):
    """Quantize 16 exact probabilities (fp64); returns (Phat fp64[16], mode)."""
    ptil = _c(ptil, np.float64)
    out = np.empty(16, np.float64)
    mode = ctypes.c_int(0)
    lib().or_p_block(_p(ptil), p_mode, p_c, tau, _p(out), ctypes.cast(ctypes.pointer(mode), ctypes.c_void_p))
    return out, mode.value


def block_sse(x, xh) -> float:
    x = _c(x, np.float32)
    xh = _c(xh, np.float32)
    return lib().or_block_sse(_p(x), _p(xh), x.size)


def fwht128(x) -> np.ndarray:
    y = np.array(x, np.float32).copy()
    lib().or_fwht128(_p(y))
    return y


def rotate128(x) -> np.ndarray:
    y = np.array(x, np.float32).copy()
    lib().or_rotate128(_p(y))
    return y


# ---- layout sizes ----------------------------------------------------------

def record_bytes(cfg: Config) -> int:
    return lib().or_record_bytes(ctypes.byref(cfg))


def qpack_stride(cfg: Config) -> int:
    return lib().or_qpack_stride(ctypes.byref(cfg))


def mem_ratio(cfg: Config) -> float:
    return lib().or_mem_ratio(ctypes.byref(cfg))


# ---- path steps ------------------------------------------------------------

def quantize_kv_pages(cfg: Config, k, v, dst_pages, mu, k_gscale: float, v_gscale: float,
                      pool: np.ndarray) -> np.ndarray:
    """k, v: uint16 [n][128][Hkv][128]; writes the records into pool (uint8) in
    place (destinations outside the pool are skipped)."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    dst = _c(dst_pages, np.int32)
    mu = _c(mu, np.float32)
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    lib().or_quantize_kv_pages(ctypes.byref(cfg), _p(k), _p(v), _p(dst), dst.size, _p(mu),
                               k_gscale, v_gscale, _p(pool))
    return pool


def quantize_query(cfg: Config, q, mu) -> np.ndarray:
    """q: uint16 [B][Hq][128] -> uint8 [B][stride]."""
    q = _c(q, np.uint16)
    mu = _c(mu, np.float32)
    B = q.shape[0]
    out = np.zeros((B, qpack_stride(cfg)), np.uint8)
    lib().or_quantize_query(ctypes.byref(cfg), _p(q), B, _p(mu), _p(out))
    return out


def decode_attention(cfg: Config, q_packed, q, mu, pool, block_table, seq_lens, sink_k, sink_v,
                     tail_k, tail_v, tau: float, k_gscale: float, v_gscale: float,
                     flags: int = 0) -> np.ndarray:
    """Returns fp64 [B][Hq][128]."""
    qp = _c(q_packed, np.uint8)
    q = _c(q, np.uint16)
    mu = _c(mu, np.float32)
    pool = _c(pool, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B = q.shape[0]
    out = np.zeros((B, cfg.num_q_heads, 128), np.float64)
    args = [_c(a, np.uint16) for a in (sink_k, sink_v, tail_k, tail_v)]
    lib().or_decode_attention(ctypes.byref(cfg), _p(qp), _p(q), _p(mu), _p(pool), _p(bt),
                              bt.shape[1] if bt.ndim == 2 else 0, _p(sl), *[_p(a) for a in args],
                              B, tau, k_gscale, v_gscale, flags, _p(out))
    return out


def attention_identity_quant(cfg: Config, q, k, v, mu) -> np.ndarray:
    """q: uint16 [Hq][128]; k, v: uint16 [L][Hkv][128] -> fp64 [Hq][128]."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    mu = _c(mu, np.float32)
    out = np.zeros((cfg.num_q_heads, 128), np.float64)
    lib().or_attention_identity_quant(ctypes.byref(cfg), _p(q), _p(k), _p(v), k.shape[0], _p(mu), _p(out))
    return out
