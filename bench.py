"""Benchmark of the NVFP4 KV-cache hot path on one GB300 (or N replicas).

Headline workload (the metric's configuration): single-sequence decode at a
131072-token context, 36 layers, 32 query / 8 KV heads, head_dim 128, full
recipe (16-token BF16 sink, Hadamard + centered keys with {4,6} scales,
two-term query, FP4 probabilities with c = 8, tau = 1.0), 128-token pages
with a shuffled physical block table.  One timed step = for each of the 36
layers, one bd_decode_attention call on the raw bf16 query (the decode kernel
quantizes it: the bytes bd_quantize_query would write), replayed as one CUDA
graph; --two-call times bd_quantize_query + bd_decode_attention instead.

The same run also times, each on its own workload and with its own clock
window, every other configuration of the workload table ("configs" in the
line): the 4096-token single-layer parity case, the page-fill writer (64
sequences x 36 layers x 8 KV heads, one freshly filled 128-token page of K and
V each; NVFP4 and MXFP4), the 32768-token decode, the 128K tau sweep
{0, 0.5, 4, 448} and the 32-sequence batch (log-uniform lengths in
[1024, 65536]; NVFP4 / MXFP4 x rotation + centering on / off), plus the
decode-token append.  --no-configs keeps only the headline.

Inputs are seeded synthetic tensors (nvfp4_kv_cache_bd_gb300.synth) resident
in HBM before timing; every decode step streams more distinct pool bytes than
L2 holds (asserted), so no explicit flush is needed.  The "e2e" figure times
the same step with all layers' queries copied in from pinned host memory and
all outputs copied out, both by bd_copy_async, inside the timed graph.
Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & packed-KV HBM GB/s (% of peak) at 128K ctx; writer tok/s"
LAYERS, HQ, HKV, D = 36, 32, 8, 128
CTX = 131072


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ctx", type=int, default=CTX)
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--tau", type=float, default=1.0)
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
    ap.add_argument("--config-steps", type=int, default=0,
                    help="timed steps of each other configuration (default: --steps, at most 100)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--two-call", action="store_true",
                    help="each layer as bd_quantize_query + bd_decode_attention on the packed query (default: one "
                         "bd_decode_attention call that quantizes the query itself)")
    return ap.parse_args()


def sm_max_mhz():
    """The maximum SM clock measured on this machine (MEASURED_PEAKS.json), else
    the GB300's nominal 2070 MHz."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if d.get("sm_max_mhz"):
            return float(d["sm_max_mhz"])
    return 2070.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t_end = time.time() + 10.0          # wait for the first sample before any timing starts
        while time.time() < t_end and self._rows() == 0:
            time.sleep(0.02)

    def _rows(self):
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def mark_begin(self):
        """Called right before a timed region: rows from here on count."""
        if self.proc is not None:
            self.windows.append([self._rows(), None])

    def mark_end(self):
        """Called right after a timed region (after its synchronize)."""
        if self.proc is not None and self.windows and self.windows[-1][1] is None:
            time.sleep(self.interval_ms / 1000.0)
            self.windows[-1][1] = self._rows()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        lines = open(self.path).read().splitlines()
        os.unlink(self.path)
        if self.windows:
            lines = [ln for a, b in self.windows if b is not None for ln in lines[a:b]]
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "timed_regions": len(self.windows),
                "interval_ms": self.interval_ms}


# ------------------------------------------------------------- workload ----

class DecodeWorkload:
    """Per-layer packed pools built by the library's own writer from seeded
    bf16 K/V (generated per layer on the GPU and freed after packing).

    lens: context lengths of the batch.  One sequence takes its pages in a
    seeded shuffle of the pool; a batch takes them round-robin across the
    sequences from one shared pool.  fmt / recipe select the scale format and
    whether keys are rotated and centered."""

    def __init__(self, lens, layers, tau, device, seed=0, fmt=0, recipe=True, two_call=False):
        import torch
        import nvfp4_kv_cache_bd_gb300 as bd
        from nvfp4_kv_cache_bd_gb300 import synth
        if isinstance(lens, int):
            lens = [lens]
        self.bd, self.torch = bd, torch
        self.two_call = two_call
        self.layers, self.tau = layers, tau
        self.B = B = len(lens)
        self.ctx = bd.Context(bd.make_config(num_layers=layers, format=fmt, rotation=int(recipe),
                                             centering=int(recipe)))
        splits = [synth.split_tokens(L) for L in lens]
        npg = [s_[1] for s_ in splits]
        self.npages = sum(npg)
        maxb = max([1] + npg)
        self.seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
        if B == 1:
            bt = synth.page_permutation(self.npages, seed, device).view(1, -1).contiguous()
        else:
            rows = [[0] * maxb for _ in range(B)]
            nxt = 0
            for rnd in range(maxb):
                for b in range(B):
                    if rnd < npg[b]:
                        rows[b][rnd] = nxt
                        nxt += 1
            bt = torch.tensor(rows, dtype=torch.int32, device=device)
        self.block_table = bt
        dst = torch.cat([bt[b, :npg[b]] for b in range(B)]) if self.npages else bt.new_zeros(0)
        self.rec = self.ctx.record_bytes
        self.pools, self.sinks, self.tails, self.gscales, self.qs = [], [], [], [], []
        for l in range(layers):
            lseed = 1000 * seed + l
            mu, mask = synth.key_mean(HKV, lseed, device)
            kv = [synth.keys_values(L, HKV, lseed if B == 1 else 64 * lseed + b, device, mu=mu, mask=mask)
                  for b, L in enumerate(lens)]
            gk, gv = synth.gscales(torch.cat([x[0] for x in kv]), torch.cat([x[1] for x in kv]), mu, recipe,
                                   recipe)
            bd.set_key_shift(self.ctx, l, mu)
            pool = torch.empty(self.ctx.pool_bytes(max(1, self.npages)), dtype=torch.uint8, device=device)
            if self.npages:
                kp = torch.cat([k[16:16 + 128 * n].view(n, 128, HKV, D) for (k, _), n in zip(kv, npg)])
                vp = torch.cat([v[16:16 + 128 * n].view(n, 128, HKV, D) for (_, v), n in zip(kv, npg)])
                bd.quantize_kv_pages(self.ctx, l, kp, vp, dst, gk, gv, pool)
                del kp, vp
            sk = torch.zeros(B, 16, HKV, D, dtype=torch.bfloat16, device=device)
            sv = torch.zeros_like(sk)
            tk = torch.zeros(B, 128, HKV, D, dtype=torch.bfloat16, device=device)
            tv = torch.zeros_like(tk)
            for b, ((n_sink, n, n_tail), (k, v)) in enumerate(zip(splits, kv)):
                sk[b, :n_sink], sv[b, :n_sink] = k[:n_sink], v[:n_sink]
                tk[b, :n_tail], tv[b, :n_tail] = k[16 + 128 * n:], v[16 + 128 * n:]
            self.pools.append(pool)
            self.sinks.append((sk, sv))
            self.tails.append((tk, tv))
            self.gscales.append((gk, gv))
            self.qs.append(synth.query(B, HQ, lseed, device))
            del kv
        torch.cuda.synchronize()
        self.qp = [torch.empty(B, self.ctx.query_packed_bytes, dtype=torch.uint8, device=device)
                   for _ in range(layers)]
        self.out = [torch.empty(B, HQ, D, dtype=torch.float32, device=device) for _ in range(layers)]
        self.ws = torch.empty(bd.decode_workspace_size(self.ctx, B, maxb) // 4 + 1, dtype=torch.float32,
                              device=device)
        self.bytes_per_layer = self.npages * HKV * 2 * self.rec

    def layer(self, l, stream=None, q=None, ev=None, out=None):
        """One layer: bd_decode_attention on the raw query, which quantizes it
        inside the decode (fused, the default), or bd_quantize_query then
        bd_decode_attention on the packed query (two_call)."""
        bd = self.bd
        q = self.qs[l] if q is None else q
        out = self.out[l] if out is None else out
        if self.two_call:
            bd.quantize_query(self.ctx, l, q, self.qp[l], stream)
        if ev is not None:
            ev[0].record()
        sk, sv = self.sinks[l]
        tk, tv = self.tails[l]
        gk, gv = self.gscales[l]
        bd.decode_attention(self.ctx, l, self.qp[l] if self.two_call else None, q, self.pools[l], self.block_table,
                            self.seq_lens, sk, sv, tk, tv, self.tau, gk, gv, out, self.ws, stream)
        if ev is not None:
            ev[1].record()

    def step(self, stream=None, evs=None):
        for l in range(self.layers):
            self.layer(l, stream, ev=None if evs is None else evs[l])

    def decode_step(self, stream=None):
        """The step without the query kernels: each layer's packed query is
        left in place by an earlier step()."""
        for l in range(self.layers):
            sk, sv = self.sinks[l]
            tk, tv = self.tails[l]
            gk, gv = self.gscales[l]
            self.bd.decode_attention(self.ctx, l, self.qp[l], self.qs[l], self.pools[l], self.block_table,
                                     self.seq_lens, sk, sv, tk, tv, self.tau, gk, gv, self.out[l], self.ws, stream)


def graphed(fn, torch):
    """Capture fn (library calls on the current stream) into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g.replay


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself on one GPU): the job's
    step time is its slowest replica's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_rate(per_step_units: float, ms_step: float, world: int) -> float:
    """Whole-job throughput of weakly scaled replicas: every rank processes
    per_step_units per step, and a step lasts the slowest rank's ms_step."""
    return world * per_step_units / (ms_step * 1e-3)


def timed(fn, steps, warmup, stream, torch, dist=None, clocks=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    if clocks is not None:
        clocks.mark_begin()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark_end()
    if dist is not None:
        dist.barrier()
    return t0.elapsed_time(t1) / steps


# ------------------------------------------------------------ CPU oracle ---

class OracleDecodeSample:
    """CPU oracle's query quantization + decode on a bounded sample of one
    layer of the workload: sample_pages FP4 pages of the 128K context plus the
    BF16 sink and tail, built once; run() times one pass and scales it to
    microseconds per full step (all pages, all layers)."""

    def __init__(self, ctx_len, sample_pages, seed=0):
        import numpy as np
        import torch
        import oracle
        from nvfp4_kv_cache_bd_gb300 import synth
        self.oracle, self.np = oracle, np
        self.cfg = cfg = oracle.make_config()
        mu, mask = synth.key_mean(HKV, seed)
        n_sink, self.npages, n_tail = synth.split_tokens(ctx_len)
        self.sample_pages = sample_pages
        self.L = L = 16 + 128 * sample_pages + n_tail
        k, v = synth.keys_values(L, HKV, seed, mu=mu, mask=mask)
        q = synth.query(1, HQ, seed)
        self.gk, self.gv = synth.gscales(k, v, mu, True, True)
        u16 = lambda t: t.contiguous().view(torch.uint16).numpy()
        self.pool = np.zeros(sample_pages * HKV * 2 * oracle.record_bytes(cfg), np.uint8)
        self.bt = np.arange(sample_pages, dtype=np.int32).reshape(1, -1)
        oracle.quantize_kv_pages(cfg, u16(k[16:16 + 128 * sample_pages].reshape(sample_pages, 128, HKV, D)),
                                 u16(v[16:16 + 128 * sample_pages].reshape(sample_pages, 128, HKV, D)), self.bt[0],
                                 mu.numpy(), self.gk, self.gv, self.pool)
        sk = torch.zeros(1, 16, HKV, D, dtype=torch.bfloat16)
        sk[0] = k[:16]
        sv = torch.zeros_like(sk)
        sv[0] = v[:16]
        tk = torch.zeros(1, 128, HKV, D, dtype=torch.bfloat16)
        tv = torch.zeros_like(tk)
        tk[0, :n_tail], tv[0, :n_tail] = k[16 + 128 * sample_pages:], v[16 + 128 * sample_pages:]
        self.args = [u16(x) for x in (q, sk, sv, tk, tv)]
        self.mu = mu.numpy()

    def describe(self):
        return (f"oracle query + decode over {self.sample_pages} of {self.npages} FP4 pages of one layer plus the "
                f"BF16 sink/tail, single thread, scaled x{self.npages}/{self.sample_pages} pages x {LAYERS} layers")

    def run(self):
        q, sk, sv, tk, tv = self.args
        t = time.perf_counter()
        qp = self.oracle.quantize_query(self.cfg, q, self.mu)
        self.oracle.decode_attention(self.cfg, qp, q, self.mu, self.pool, self.bt, self.np.array([self.L], self.np.int32),
                                     sk, sv, tk, tv, 1.0, self.gk, self.gv)
        dt = time.perf_counter() - t
        return dt * 1e6 * (self.npages / self.sample_pages) * LAYERS, dt


def _oracle_all_cores_worker(args):
    """One process of the all-core oracle run: build a sample, wait for the
    others, time one pass."""
    ctx_len, pages, barrier = args
    smp = OracleDecodeSample(ctx_len, pages)
    barrier.wait()
    t = time.perf_counter()
    smp.run()
    return time.perf_counter() - t


def oracle_extra_baselines(ctx_len):
    """More oracle timings on the host: the page-fill writer (1 thread), the
    4096-token single-layer step (1 thread), and the decode sample run by
    every host core at once (one process each, spawned)."""
    import multiprocessing as mp
    import numpy as np
    import torch
    import oracle
    from nvfp4_kv_cache_bd_gb300 import synth
    out = {}
    cfg = oracle.make_config()
    pages = 16
    mu, mask = synth.key_mean(HKV, 1)
    k, v = synth.keys_values(128 * pages, HKV, 1, mu=mu, mask=mask)
    u16 = lambda t: t.contiguous().view(torch.uint16).numpy()
    pool = np.zeros(pages * HKV * 2 * oracle.record_bytes(cfg), np.uint8)
    t = time.perf_counter()
    oracle.quantize_kv_pages(cfg, u16(k.view(pages, 128, HKV, D)), u16(v.view(pages, 128, HKV, D)),
                             np.arange(pages, dtype=np.int32), mu.numpy(), 1.0, 1.0, pool)
    dt = time.perf_counter() - t
    out["writer_tok_per_s_1core"] = pages * 128 / dt
    smp0 = OracleDecodeSample(4096, 31)
    out["step_4096_ctx_1_layer_us_1core"] = smp0.run()[1] * 1e6
    ncores = max(1, os.cpu_count() or 1)
    spages = 64
    c = mp.get_context("spawn")
    barrier = c.Manager().Barrier(ncores)
    with c.Pool(ncores) as pool_:
        dts = pool_.map(_oracle_all_cores_worker, [(ctx_len, spages, barrier)] * ncores)
    npages = synth.split_tokens(ctx_len)[1]
    out["decode_step_us_all_cores"] = max(dts) / ncores * 1e6 * (npages / spages) * LAYERS
    out["all_cores"] = ncores
    out["all_cores_sample"] = (f"{ncores} processes at once, each the oracle query + decode over {spages} of {npages} "
                               "pages of one layer; step time = slowest process / processes, scaled to all pages "
                               f"and {LAYERS} layers")
    return out


# -------------------------------------------------------------- reference --

def run_reference(args):
    """The oracle, as it stands, timed on the host cores: each step is one
    bounded sample of the decode workload scaled to a full step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = OracleDecodeSample(args.ctx, 256)
    samples = []
    for i in range(args.warmup + args.steps):
        us, _ = smp.run()
        if i >= args.warmup:
            samples.append(us)
    v = statistics.median(samples)
    line = {"metric": METRIC, "value": v, "unit": "µs/step", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": v / 1000.0, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 attention / f32 quantizer", "data": "synthetic", "impl": "reference",
            "config": {"workload": f"decode {args.ctx}-token ctx, batch 1, {LAYERS} layers, 32q/8kv heads, d128, "
                                   "NVFP4 full recipe, tau 1.0", "global_batch": 1, "seq_len": args.ctx,
                       "parallelism": "single host thread"},
            "cpu_baseline": {"value": v, "unit": "µs/step", "cores": 1, "kind": "oracle", "sample": smp.describe()},
            "e2e": {"value": v, "unit": "µs/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- native --

L2_BYTES = 129 * 1024 * 1024


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist
    import nvfp4_kv_cache_bd_gb300 as bd
    from nvfp4_kv_cache_bd_gb300 import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    build.build_library()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    stream = torch.cuda.current_stream()
    hbm_peak, peak_src = peaks()
    clocks = ClockSampler(local)
    clocks.start()
    cfg_steps = args.config_steps or min(args.steps, 100)

    # ---------------- decode workload (headline)
    wl = DecodeWorkload(args.ctx, args.layers, args.tau, device, seed=rank, two_call=args.two_call)
    step_bytes = wl.bytes_per_layer * args.layers
    assert step_bytes > L2_BYTES, "a step must stream more than L2 holds"
    fn = graphed(lambda: wl.step(), torch)   # one step = 36 x (query quantization + decode)
    ms = timed(fn, args.steps, args.warmup, stream, torch, pg, clocks)
    if args.two_call:
        # the decode alone inside a graphed step (packed queries left by the
        # step above): its per-layer time is the decode launch's in-step duration
        dec_graph_ms = timed(graphed(lambda: wl.decode_step(), torch), args.steps, args.warmup, stream, torch, pg,
                             clocks)
    else:
        dec_graph_ms = ms   # the step is the layers' decode calls alone
    # stream-ordered, one decode call at a time with events around it
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.layers)]
    durs = []
    for _ in range(10):
        wl.step(evs=evs)
        torch.cuda.synchronize()
        durs += [a_.elapsed_time(b_) for a_, b_ in evs]
    err = bd.read_device_error(wl.ctx)
    if err != bd.OK:
        raise RuntimeError(f"device error word: {bd.status_string(err)}")
    ms = max_over_ranks(ms, pg, device)
    dec_graph_ms = max_over_ranks(dec_graph_ms, pg, device)
    us_step = ms * 1000.0
    call_ms = statistics.mean(durs)
    in_step_ms = dec_graph_ms / args.layers
    achieved_in_step = wl.bytes_per_layer / (in_step_ms * 1e-3) / 1e9
    achieved_call = wl.bytes_per_layer / (call_ms * 1e-3) / 1e9

    # ---------------- end to end through the C ABI with host buffers: one
    # host->device copy of the step's queries (all layers) from pinned memory,
    # the layers, one device->host copy of the step's outputs; both copies by
    # bd_copy_async, a kernel that reads and writes the pinned host buffers
    # over the CPU-GPU link
    q_host = torch.stack([q for q in wl.qs]).cpu().pin_memory()          # [layers][1][Hq][D] bf16
    out_host = torch.empty(args.layers, 1, HQ, D, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q_host, device=device)
    out_dev = torch.empty(args.layers, 1, HQ, D, dtype=torch.float32, device=device)

    def e2e_step():
        bd.copy_async(q_dev, q_host)
        for l in range(args.layers):
            wl.layer(l, q=q_dev[l], out=out_dev[l])
        bd.copy_async(out_host, out_dev)

    e2e_ms = timed(graphed(e2e_step, torch), args.steps, args.warmup, stream, torch, pg, clocks)
    e2e_ms = max_over_ranks(e2e_ms, pg, device)
    h2d = q_host.numel() * q_host.element_size()
    d2h = out_host.numel() * out_host.element_size()

    configs = None
    if not args.no_configs:
        configs = {}
        gbs = step_bytes / (ms * 1e-3) / 1e9
        sweep = {str(args.tau): {"us_per_step": us_step, "packed_kv_gbs": gbs, "frac_of_peak": gbs / hbm_peak,
                                 "packed_bytes_per_step": step_bytes, "note": "the headline measurement"}}
        for tau in (0.0, 0.5, 4.0, 448.0):
            wl.tau = tau
            sweep[str(tau)] = step_rate(wl, cfg_steps, args.warmup, stream, torch, pg, hbm_peak, clocks)
        wl.tau = args.tau
        configs[f"decode_{args.ctx // 1024}k_ctx_{args.layers}_layers_tau_sweep"] = sweep
    del wl
    torch.cuda.empty_cache()

    writer = bench_writer(args, device, stream, torch, bd, pg, hbm_peak, clocks=clocks)
    if configs is not None:
        configs.update(run_configs(args, device, stream, torch, bd, pg, hbm_peak, clocks, cfg_steps))
    clk = clocks.stop()

    line = {
        "metric": METRIC, "value": us_step, "unit": "µs/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 operands, f16 mma, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"decode {args.ctx}-token ctx, batch 1, {args.layers} layers, 32q/8kv heads, d128, "
                               f"NVFP4 full recipe, tau {args.tau}, shuffled 128-token pages",
                   "global_batch": world, "seq_len": args.ctx, "layers": args.layers,
                   "l2": f"not flushed: each step streams {args.layers} distinct layers' pools "
                         f"({step_bytes / 1e9:.2f} GB) >> 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "packed_kv_gbs": job_rate(step_bytes, ms, world) / 1e9,
        "packed_kv_frac_of_peak": job_rate(step_bytes, ms, world) / 1e9 / (hbm_peak * world),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (one bd_decode_attention call"
                               + (")" if args.two_call else ", query quantization inside)"),
                     "achieved": achieved_in_step, "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved_in_step / hbm_peak,
                     "frac_basis": (f"in step: one graph of the {args.layers} layers' decode calls alone"
                                    + (" (packed queries in place)" if args.two_call else "")
                                    + f", {dec_graph_ms * 1000:.1f} us / {args.layers} = "
                                    f"{in_step_ms * 1000:.2f} us per call"),
                     "frac_in_step": achieved_in_step / hbm_peak, "us_per_call_in_step": in_step_ms * 1000,
                     "frac_call": achieved_call / hbm_peak, "achieved_call": achieved_call,
                     "us_per_call_alone": call_ms * 1000,
                     "traffic": decode_traffic(args), "bytes_per_launch": wl_bytes_note(args)},
        "e2e": {"value": e2e_ms * 1000.0, "unit": "µs/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # per layer: bd_decode_attention's one decode kernel (splits merged and,
        # unless --two-call, the query quantized inside it); --two-call adds
        # the query kernel
        "gpu_launches": args.steps * args.layers * (2 if args.two_call else 1),
        "launch": (f"one CUDA graph per step ({args.layers} x "
                   + ("query kernel + decode kernel" if args.two_call else "decode kernel") +
                   ", programmatic dependent launch)"),
        "clocks": clk,
        "writer": writer,
    }
    if configs is not None:
        line["configs"] = configs
    if rank == 0 and not args.no_cpu_baseline:
        smp = OracleDecodeSample(args.ctx, 256)
        runs = [smp.run() for _ in range(3)]
        line["cpu_baseline"] = {"value": statistics.median(r[0] for r in runs), "unit": "µs/step", "cores": 1,
                                "kind": "oracle",
                                "sample": smp.describe() + f"; median of 3 runs of {runs[0][1]:.1f} s"}
        line["cpu_baseline"].update(oracle_extra_baselines(args.ctx))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        dist.barrier()
        dist.destroy_process_group()


# DRAM bytes (read + write) of one decode_kernel launch on the 131072-token
# context, from ncu (dram__bytes_read.sum + dram__bytes_write.sum) on a 2-layer
# run of this bench; a launch's traffic does not depend on the layer count.
# Valid only for the kernel code it was taken on: reported as null once the
# hash of that code (comments and whitespace left out) differs.
DECODE_TRAFFIC = {"sources_sha256_16": "7656eab6e85792c2", "ctx": 131072, "bytes": 151523328 + 3516160}
DECODE_SOURCES = ("bd_decode.cu", "bd_device.cuh", "bd_internal.h", "bd_query.cuh")
# Warp instructions one NVFP4 writer launch of the writer bench executes
# (ncu smsp__inst_executed.sum, profiles/writer_kernel_64seq_page_fill.md),
# for the writer's issue-rate roofline; null once its code changes.
WRITER_INSTR = {"sources_sha256_16": "1f89f52f52ebd7a2", "fmt": 0, "warp_instructions": 10993664}
WRITER_SOURCES = ("bd_writer.cu", "bd_device.cuh", "bd_internal.h")


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs folded to one
    space: two sources with the same code_only text compile alike."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def sources_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "nvfp4_kv_cache_bd_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def decode_sources_hash():
    return sources_hash(DECODE_SOURCES)


def decode_traffic(args):
    if decode_sources_hash() != DECODE_TRAFFIC["sources_sha256_16"] or args.ctx != DECODE_TRAFFIC["ctx"]:
        return None
    return DECODE_TRAFFIC["bytes"]


def step_rate(wl, steps, warmup, stream, torch, pg, hbm_peak, clocks=None):
    """µs per step of a graphed decode step and its packed-KV bandwidth."""
    ms = timed(graphed(lambda: wl.step(), torch), steps, warmup, stream, torch, pg, clocks)
    ms = max_over_ranks(ms, pg, torch.device("cuda", torch.cuda.current_device()))
    gbs = wl.bytes_per_layer * wl.layers / (ms * 1e-3) / 1e9
    return {"us_per_step": ms * 1000.0, "packed_kv_gbs": gbs, "frac_of_peak": gbs / hbm_peak,
            "packed_bytes_per_step": wl.bytes_per_layer * wl.layers}


def bench_append(args, device, stream, torch, bd, pg, hbm_peak, clocks=None):
    """bd_append_kv for 64 sequences per layer: a step of 36 launches with no
    page completed, and one where every sequence completes a page (once
    every 128 decode steps)."""
    from nvfp4_kv_cache_bd_gb300 import synth
    B, layers = 64, args.layers
    ctx = bd.Context(bd.make_config(num_layers=layers))
    mu, _ = synth.key_mean(HKV, 6000, device)
    st = []
    for l in range(layers):
        bd.set_key_shift(ctx, l, mu)
        g = torch.Generator(device=device)
        g.manual_seed(6000 + l)
        st.append(dict(
            sk=torch.randn(B, 16, HKV, D, generator=g, device=device).to(torch.bfloat16),
            sv=torch.randn(B, 16, HKV, D, generator=g, device=device).to(torch.bfloat16),
            tk=torch.randn(B, 128, HKV, D, generator=g, device=device).to(torch.bfloat16),
            tv=torch.randn(B, 128, HKV, D, generator=g, device=device).to(torch.bfloat16),
            kn=torch.randn(B, HKV, D, generator=g, device=device).to(torch.bfloat16),
            vn=torch.randn(B, HKV, D, generator=g, device=device).to(torch.bfloat16),
            pool=torch.empty(ctx.pool_bytes(2 * B), dtype=torch.uint8, device=device)))
    bt = torch.arange(2 * B, dtype=torch.int32, device=device).view(B, 2)
    out = {}
    for name, L in (("no_page_completed", 16 + 128 + 5), ("every_sequence_completes_a_page", 16 + 128 + 127)):
        sl = torch.full((B,), L, dtype=torch.int32, device=device)

        def step():
            for l in range(layers):
                t = st[l]
                bd.append_kv(ctx, l, t["kn"], t["vn"], sl, bt, t["sk"], t["sv"], t["tk"], t["tv"], 1.0, 1.0,
                             t["pool"])

        ms = timed(graphed(step, torch), 100, args.warmup, stream, torch, pg, clocks)
        out[name + "_us_per_step"] = ms * 1000.0
    out["workload"] = f"{B} sequences x {layers} layers, one token each"
    out["page_fill_tok_per_s"] = B * 128 / (out["every_sequence_completes_a_page_us_per_step"] * 1e-6)
    return out


def run_configs(args, device, stream, torch, bd, pg, hbm_peak, clocks, steps):
    """The other configurations of the workload table, each a full step."""
    from nvfp4_kv_cache_bd_gb300 import synth
    out = {}
    wl = DecodeWorkload(4096, 1, 1.0, device, two_call=args.two_call)
    r = step_rate(wl, steps, args.warmup, stream, torch, pg, hbm_peak, clocks)
    r["note"] = ("4096-token context, 1 layer (the parity configuration): 4.6 MB of packed K/V, inside L2, so this "
                 "is a latency figure, not a bandwidth one")
    out["decode_4k_ctx_1_layer"] = r
    del wl
    out["writer_mxfp4"] = bench_writer(args, device, stream, torch, bd, pg, hbm_peak, fmt=1, clocks=clocks)
    wl = DecodeWorkload(32768, args.layers, 1.0, device, two_call=args.two_call)
    assert wl.bytes_per_layer * wl.layers > L2_BYTES
    out[f"decode_32k_ctx_{args.layers}_layers"] = step_rate(wl, steps, args.warmup, stream, torch, pg, hbm_peak,
                                                            clocks)
    del wl
    torch.cuda.empty_cache()
    lens = synth.log_uniform_lengths(32, 1024, 65536, 0)
    batch = {"lengths": "32 seqs, log-uniform in [1024, 65536], %d tokens in all" % sum(lens)}
    for fmt, fname in ((0, "nvfp4"), (1, "mxfp4")):
        for recipe in (True, False):
            wl = DecodeWorkload(lens, args.layers, 1.0, device, fmt=fmt, recipe=recipe, two_call=args.two_call)
            batch[f"{fname}_{'rotation_centering' if recipe else 'plain_keys'}"] = step_rate(
                wl, steps, args.warmup, stream, torch, pg, hbm_peak, clocks)
            del wl
            torch.cuda.empty_cache()
    out[f"decode_batch_32_{args.layers}_layers"] = batch
    out["append"] = bench_append(args, device, stream, torch, bd, pg, hbm_peak, clocks)
    return out


def wl_bytes_note(args):
    npages = (args.ctx - 16) // 128
    return npages * HKV * 2 * 9216


def bench_writer(args, device, stream, torch, bd, pg, hbm_peak, fmt=0, clocks=None):
    from nvfp4_kv_cache_bd_gb300 import synth
    seqs, layers = 64, args.layers
    ctx = bd.Context(bd.make_config(num_layers=layers, format=fmt))
    pools, ks, vs, gs = [], [], [], []
    dst = synth.page_permutation(seqs, 7, device)
    for l in range(layers):
        mu, mask = synth.key_mean(HKV, 5000 + l, device)
        k, v = synth.keys_values(seqs * 128, HKV, 5000 + l, device, mu=mu, mask=mask)
        bd.set_key_shift(ctx, l, mu)
        gs.append(synth.gscales(k, v, mu, True, True))
        ks.append(k.view(seqs, 128, HKV, D))
        vs.append(v.view(seqs, 128, HKV, D))
        pools.append(torch.empty(ctx.pool_bytes(seqs), dtype=torch.uint8, device=device))

    def step():
        for l in range(layers):
            bd.quantize_kv_pages(ctx, l, ks[l], vs[l], dst, gs[l][0], gs[l][1], pools[l])

    ms = timed(graphed(step, torch), args.steps, args.warmup, stream, torch, pg, clocks)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(layers)]
    durs = []
    for _ in range(3):
        for l in range(layers):
            evs[l][0].record()
            bd.quantize_kv_pages(ctx, l, ks[l], vs[l], dst, gs[l][0], gs[l][1], pools[l])
            evs[l][1].record()
        torch.cuda.synchronize()
        durs += [a.elapsed_time(b) for a, b in evs]
    ms = max_over_ranks(ms, pg, device)
    call_bytes = seqs * 128 * HKV * D * 2 * 2 + seqs * HKV * 2 * ctx.record_bytes
    call_ms = statistics.mean(durs)
    tok = seqs * 128
    fmt_name = "NVFP4" if fmt == 0 else "MXFP4"
    out = {"workload": f"{seqs} seqs x {layers} layers x 8 kv heads, one 128-token page of K and V each, {fmt_name}",
           "tok_per_s": job_rate(tok, ms, pg.get_world_size() if pg is not None else 1),
           "ms_per_step": ms, "gpu_launches_per_step": layers,
           "roofline": {"bound": "hbm", "kernel": "writer_kernel", "achieved": call_bytes / (call_ms * 1e-3) / 1e9,
                        "peak": hbm_peak, "unit": "GB/s", "frac": call_bytes / (call_ms * 1e-3) / 1e9 / hbm_peak,
                        "bytes_per_launch": call_bytes}}
    # The writer is bound by instruction issue, not by HBM: the same launch
    # against the SMs' issue rate (one warp instruction per scheduler and
    # cycle: SMs x 4 x the maximum SM clock), on its in-step duration.
    if fmt == WRITER_INSTR["fmt"] and sources_hash(WRITER_SOURCES) == WRITER_INSTR["sources_sha256_16"]:
        props = torch.cuda.get_device_properties(device)
        mhz = sm_max_mhz()
        peak = props.multi_processor_count * 4 * mhz * 1e6 / 1e12
        step_launch_s = ms * 1e-3 / layers
        ach = WRITER_INSTR["warp_instructions"] / step_launch_s / 1e12
        out["roofline_issue"] = {"bound": "alu", "kernel": "writer_kernel", "achieved": ach, "peak": peak,
                                 "unit": "T warp instructions/s", "frac": ach / peak,
                                 "warp_instructions_per_launch": WRITER_INSTR["warp_instructions"],
                                 "basis": f"{props.multi_processor_count} SMs x 4 schedulers x {mhz:.0f} MHz; "
                                          "in-step launch time (step / layers)"}
    return out


if __name__ == "__main__":
    main()
