"""bd_copy_async on the GPU: bytes moved between pinned host memory and
device memory (both directions, and device to device) by the copy kernel,
compared bit for bit, for sizes around the 16-byte word and the grid; and
the arguments it refuses before launching anything."""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_bd_gb300 as bd

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 17, 4096 + 5, 1 << 20, (3 << 20) + 9]


@pytest.mark.parametrize("nbytes", SIZES)
def test_host_device_round_trip(nbytes):
    rng = np.random.default_rng(nbytes)
    host = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    dev2 = torch.full((nbytes,), 0x3C, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    bd.copy_async(dev, host)        # host -> device
    bd.copy_async(dev2, dev)        # device -> device
    bd.copy_async(back, dev2)       # device -> host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)
    assert torch.equal(back, host)


def test_copy_captured_in_a_graph():
    """The bench's end-to-end step captures the copies into a CUDA graph."""
    host = torch.arange(4096, dtype=torch.float32).pin_memory()
    dev = torch.zeros(4096, dtype=torch.float32, device="cuda")
    out = torch.zeros(4096, dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bd.copy_async(dev, host)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bd.copy_async(dev, host)
        dev.mul_(2.0)
        bd.copy_async(out, dev)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, host * 2.0)


def test_refused_arguments_launch_nothing():
    L = bd.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dev = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(1024, dtype=torch.uint8)           # not pinned: the GPU may not touch it
    pinned = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    P = ctypes.c_void_p
    assert L.bd_copy_async(P(pageable.data_ptr()), P(dev.data_ptr()), 1024, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(dev.data_ptr()), P(pageable.data_ptr()), 1024, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(dev.data_ptr() + 8), P(pinned.data_ptr()), 64, s) == bd.ERR_INVALID_ARG
    assert L.bd_copy_async(P(dev.data_ptr()), P(dev.data_ptr() + 16), 64, s) == bd.ERR_INVALID_ARG
    # a range that runs past the end of its allocation into unknown memory
    assert L.bd_copy_async(P(pinned.data_ptr()), P(dev.data_ptr()), 1 << 40, s) == bd.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(dev).item() == 0 and torch.count_nonzero(pinned).item() == 0
    with pytest.raises(ValueError):
        bd.copy_async(dev, pageable)
