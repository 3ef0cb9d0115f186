"""Oracle work for the full-size parity tests, spread over CPU processes.

The oracle is page-local for the writer (a record depends on its own page
only) and sequence-local for the decode, so pages and sequences are split
across a process pool.  The pool uses the "spawn" start method: a process
forked after the parent has touched CUDA can hang.  Inputs reach the workers
as memory-mapped .npy files; each worker returns only its own records or
outputs.  Worker functions live at module level so spawned processes can
import them.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

import oracle

H, HQ, D = 8, 32, 128


def _cfg(kw):
    return oracle.make_config(**kw)


def _writer_slice(args):
    kw, kpath, vpath, mupath, lo, hi, gk, gv = args
    cfg = _cfg(kw)
    k = np.load(kpath, mmap_mode="r")[lo:hi]
    v = np.load(vpath, mmap_mode="r")[lo:hi]
    mu = np.load(mupath)
    n = hi - lo
    pool = np.zeros(n * H * 2 * oracle.record_bytes(cfg), np.uint8)
    oracle.quantize_kv_pages(cfg, np.ascontiguousarray(k), np.ascontiguousarray(v), np.arange(n, dtype=np.int32), mu,
                             gk, gv, pool)
    return lo, pool


def _decode_slice(args):
    (kw, qp, q, mu, pool_path, bt, sl, sk, sv, tk, tv, tau, gk, gv) = args
    pool = np.load(pool_path, mmap_mode="r")
    return oracle.decode_attention(_cfg(kw), qp, q, mu, np.ascontiguousarray(pool), bt, sl, sk, sv, tk, tv, tau, gk,
                                   gv)


class OraclePool:
    """A spawn-context process pool plus a scratch directory for inputs."""

    def __init__(self, procs: int | None = None):
        n = procs or max(1, min(16, (os.cpu_count() or 2)))
        self.procs = n
        self.pool = mp.get_context("spawn").Pool(n)
        self.dir = tempfile.TemporaryDirectory()

    def close(self):
        self.pool.close()
        self.pool.join()
        self.dir.cleanup()

    def _save(self, name, arr):
        path = os.path.join(self.dir.name, name + ".npy")
        np.save(path, arr)
        return path

    def quantize_pages(self, kw: dict, k_pages: np.ndarray, v_pages: np.ndarray, dst: np.ndarray, mu: np.ndarray,
                       gk: float, gv: float, pool: np.ndarray):
        """oracle.quantize_kv_pages over all pages, written into pool at dst."""
        n = k_pages.shape[0]
        if n == 0:
            return pool
        kp, vp, mp_ = self._save("k", k_pages), self._save("v", v_pages), self._save("mu", mu)
        step = max(1, -(-n // (4 * self.procs)))
        jobs = [(kw, kp, vp, mp_, lo, min(n, lo + step), gk, gv) for lo in range(0, n, step)]
        cfg = _cfg(kw)
        rec = oracle.record_bytes(cfg)
        per_page = H * 2 * rec
        for lo, part in self.pool.imap_unordered(_writer_slice, jobs):
            for i in range(part.size // per_page):
                phys = int(dst[lo + i])
                pool[phys * per_page:(phys + 1) * per_page] = part[i * per_page:(i + 1) * per_page]
        return pool

    def decode(self, kw: dict, qp, q, mu, pool, block_table, seq_lens, sink_k, sink_v, tail_k, tail_v, tau, gk, gv):
        """oracle.decode_attention, one sequence per job."""
        pool_path = self._save("pool", pool)
        B = len(seq_lens)
        jobs = [(kw, qp[b:b + 1], q[b:b + 1], mu, pool_path, block_table[b:b + 1], seq_lens[b:b + 1],
                 sink_k[b:b + 1], sink_v[b:b + 1], tail_k[b:b + 1], tail_v[b:b + 1], tau, gk, gv) for b in range(B)]
        return np.concatenate(self.pool.map(_decode_slice, jobs), axis=0)
