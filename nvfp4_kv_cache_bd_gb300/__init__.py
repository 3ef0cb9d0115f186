"""GB300 (sm_103a) NVFP4 KV-cache hot path: page-fill writer, two-term FP4
query quantizer and paged FP4 decode attention.

Thin Python binding over the C ABI in ``include/bd.h`` (``libbd.so``, built
in-tree by ``nvfp4_kv_cache_bd_gb300.build``).  Functions keep the C names
without the ``bd_`` prefix and only marshal arguments: every step of the path
runs in the library's CUDA kernels.  PyTorch provides device memory and
streams.  Importing works without a GPU; the calls raise if the library is
missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

FORMAT_NVFP4, FORMAT_MXFP4 = 0, 1
P_NONE, P_AMAX6, P_AMAX2_OR_AMAX6 = 0, 1, 2

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5


class BDError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "sink_tokens", "format",
        "key_search", "rotation", "centering", "query_terms", "p_mode", "p_c", "pool_pages")]


def make_config(num_layers=1, num_q_heads=32, num_kv_heads=8, format=FORMAT_NVFP4, key_search=1, rotation=1,
                centering=1, query_terms=2, p_mode=P_AMAX2_OR_AMAX6, p_c=8, head_dim=128, page_size=128,
                sink_tokens=16, pool_pages=0) -> Config:
    return Config(num_layers, num_q_heads, num_kv_heads, head_dim, page_size, sink_tokens, format, key_search,
                  rotation, centering, query_terms, p_mode, p_c, pool_pages)


EXPORTS = ("bd_create", "bd_destroy", "bd_status_string", "bd_set_key_shift", "bd_record_bytes",
           "bd_query_packed_bytes", "bd_quantize_kv_pages", "bd_append_kv", "bd_quantize_query",
           "bd_decode_workspace_size",
           "bd_decode_attention", "bd_decode_attention_noalloc", "bd_read_device_error",
           "bd_selftest_bounded_wait", "bd_copy_async")

_lib = None


def lib() -> ctypes.CDLL:
    """Load libbd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it with `python -m nvfp4_kv_cache_bd_gb300.build`")
        L = ctypes.CDLL(LIB)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        CP = ctypes.POINTER(Config)
        sig = {
            "bd_create": (I, [CP, ctypes.POINTER(P)]),
            "bd_destroy": (None, [P]),
            "bd_status_string": (ctypes.c_char_p, [I]),
            "bd_set_key_shift": (I, [P, I, P]),
            "bd_record_bytes": (SZ, [P]),
            "bd_query_packed_bytes": (SZ, [P]),
            "bd_quantize_kv_pages": (I, [P, I, P, P, P, I, F, F, P, P]),
            "bd_append_kv": (I, [P, I, P, P, P, P, I, P, P, P, P, I, F, F, P, P]),
            "bd_quantize_query": (I, [P, I, P, I, P, P]),
            "bd_decode_workspace_size": (SZ, [P, I, I]),
            "bd_decode_attention": (I, [P, I, P, P, P, P, I, P, P, P, P, P, I, F, F, F, P, P, SZ, P]),
            "bd_decode_attention_noalloc": (I, [P, I, P, P, P, P, I, P, P, P, P, P, I, F, F, F, P, P]),
            "bd_read_device_error": (I, [P, P, ctypes.POINTER(I)]),
            "bd_selftest_bounded_wait": (I, [P, I, P]),
            "bd_copy_async": (I, [P, P, SZ, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().bd_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise BDError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Context:
    """Owns a bd_ctx (bd_create / bd_destroy)."""

    def __init__(self, cfg: Config):
        h = ctypes.c_void_p()
        _check(lib().bd_create(ctypes.byref(cfg), ctypes.byref(h)), "bd_create")
        self.handle = h
        self.cfg = cfg

    def close(self):
        if self.handle:
            lib().bd_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def record_bytes(self) -> int:
        return lib().bd_record_bytes(self.handle)

    @property
    def query_packed_bytes(self) -> int:
        return lib().bd_query_packed_bytes(self.handle)

    def pool_bytes(self, num_pages: int) -> int:
        return num_pages * self.cfg.num_kv_heads * 2 * self.record_bytes


def set_key_shift(ctx: Context, layer: int, mu: torch.Tensor):
    mu = mu.detach().to("cpu", torch.float32).contiguous()
    _check(lib().bd_set_key_shift(ctx.handle, layer, _ptr(mu)), "bd_set_key_shift")


def quantize_kv_pages(ctx: Context, layer: int, k, v, dst_pages, k_gscale: float, v_gscale: float, kv_pool,
                      stream=None):
    n = 0 if k is None else k.shape[0]
    if n:
        _dev(k, "k", torch.bfloat16)
        _dev(v, "v", torch.bfloat16)
        _dev(dst_pages, "dst_pages", torch.int32)
        _dev(kv_pool, "kv_pool", torch.uint8)
    _check(lib().bd_quantize_kv_pages(ctx.handle, layer, _ptr(k), _ptr(v), _ptr(dst_pages), n, k_gscale, v_gscale,
                                      _ptr(kv_pool), _stream(stream)), "bd_quantize_kv_pages")


def append_kv(ctx: Context, layer: int, k_new, v_new, seq_lens, block_table, sink_k, sink_v, tail_k, tail_v,
              k_gscale: float, v_gscale: float, kv_pool, stream=None):
    """bd_append_kv: store each sequence's new token at position seq_lens[b]
    and pack the tail page it completes into the pool."""
    B = k_new.shape[0]
    max_blocks = block_table.shape[1] if block_table is not None and block_table.dim() == 2 else 0
    if B:
        _dev(k_new, "k_new", torch.bfloat16)
        _dev(v_new, "v_new", torch.bfloat16)
        _dev(seq_lens, "seq_lens", torch.int32)
        for t, nme in ((sink_k, "sink_k"), (sink_v, "sink_v"), (tail_k, "tail_k"), (tail_v, "tail_v")):
            _dev(t, nme, torch.bfloat16)
    _check(lib().bd_append_kv(ctx.handle, layer, _ptr(k_new), _ptr(v_new), _ptr(seq_lens), _ptr(block_table),
                              max_blocks, _ptr(sink_k), _ptr(sink_v), _ptr(tail_k), _ptr(tail_v), B, k_gscale,
                              v_gscale, _ptr(kv_pool), _stream(stream)), "bd_append_kv")


def quantize_query(ctx: Context, layer: int, q, q_packed, stream=None):
    B = q.shape[0]
    if B:
        _dev(q, "q", torch.bfloat16)
        _dev(q_packed, "q_packed", torch.uint8)
    _check(lib().bd_quantize_query(ctx.handle, layer, _ptr(q), B, _ptr(q_packed), _stream(stream)),
           "bd_quantize_query")


def decode_workspace_size(ctx: Context, B: int, max_blocks: int) -> int:
    return lib().bd_decode_workspace_size(ctx.handle, B, max_blocks)


def decode_attention(ctx: Context, layer: int, q_packed, q, kv_pool, block_table, seq_lens, sink_k, sink_v,
                     tail_k, tail_v, tau: float, k_gscale: float, v_gscale: float, out, ws, stream=None):
    B = q.shape[0]
    max_blocks = block_table.shape[1] if block_table is not None and block_table.dim() == 2 else 0
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().bd_decode_attention(ctx.handle, layer, _ptr(q_packed), _ptr(q), _ptr(kv_pool), _ptr(block_table),
                                     max_blocks, _ptr(seq_lens), _ptr(sink_k), _ptr(sink_v), _ptr(tail_k),
                                     _ptr(tail_v), B, tau, k_gscale, v_gscale, _ptr(out), _ptr(ws), ws_bytes,
                                     _stream(stream)), "bd_decode_attention")


def decode_attention_noalloc(ctx: Context, layer: int, q_packed, q, kv_pool, block_table, seq_lens, sink_k, sink_v,
                             tail_k, tail_v, tau: float, k_gscale: float, v_gscale: float, out, stream=None):
    """bd_decode_attention_noalloc: the decode without a caller workspace and
    without device allocation, for callers that cannot allocate GPU memory
    (its scratch is a fixed 4 MiB array inside the library)."""
    B = q.shape[0]
    max_blocks = block_table.shape[1] if block_table is not None and block_table.dim() == 2 else 0
    _check(lib().bd_decode_attention_noalloc(ctx.handle, layer, _ptr(q_packed), _ptr(q), _ptr(kv_pool),
                                             _ptr(block_table), max_blocks, _ptr(seq_lens), _ptr(sink_k), _ptr(sink_v),
                                             _ptr(tail_k), _ptr(tail_v), B, tau, k_gscale, v_gscale, _ptr(out),
                                             _stream(stream)), "bd_decode_attention_noalloc")


def read_device_error(ctx: Context, stream=None) -> int:
    out = ctypes.c_int(0)
    _check(lib().bd_read_device_error(ctx.handle, _stream(stream), ctypes.byref(out)), "bd_read_device_error")
    return out.value


def copy_async(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """bd_copy_async: copy src's bytes into dst by a kernel; each tensor is a
    contiguous CUDA tensor or a contiguous pinned CPU tensor (same byte size)."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(lib().bd_copy_async(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "bd_copy_async")


def selftest_bounded_wait(ctx: Context, timeout_us: int, stream=None):
    _check(lib().bd_selftest_bounded_wait(ctx.handle, timeout_us, _stream(stream)), "bd_selftest_bounded_wait")
