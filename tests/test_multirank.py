"""The multi-GPU path of the benchmark is replicas: every rank runs its own
decode and the job's step time is the slowest rank's.  Its host logic runs
here on two CPU ranks over gloo (no GPU): the max-over-ranks reduction and
the whole-job rate of weakly scaled replicas."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")          # rank r took 1 + r ms
    rate = bench.job_rate(1000.0, ms, dist.get_world_size())
    out[rank] = (ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step_and_the_job_rate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 2.0                                   # the slower rank's step
    assert rate == pytest.approx(2 * 1000.0 / 2e-3)   # both ranks' units over the slowest step


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_rate(10.0, 2.0, 1) == pytest.approx(5000.0)
