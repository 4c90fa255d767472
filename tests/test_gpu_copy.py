"""pa_copy on the GPU: kernel copies between pinned host memory and the device, bit for bit,
also inside a replayed CUDA graph; addresses the device cannot reach are refused."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PA_ERR_INVALID_ARG = 1


def _bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", [16, 17408, 12288, 1 << 20])
def test_copy_host_device_round_trip(cuda_lib, n):
    pa = cuda_lib
    src_h = _bytes(n, n).pin_memory()
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    pa.copy(dev, src_h)
    dev2 = torch.empty_like(dev)
    pa.copy(dev2, dev)              # device to device
    pa.copy(back, dev2)             # device to host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src_h)
    assert torch.equal(back, src_h)


def test_copy_inside_a_replayed_graph_sees_each_steps_data(cuda_lib):
    pa = cuda_lib
    n = 17408
    host_in = torch.zeros(n, dtype=torch.uint8).pin_memory()
    host_out = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.copy(dev, host_in)       # warm-up outside capture
        pa.copy(host_out, dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.copy(dev, host_in)
        dev.add_(1)
        pa.copy(host_out, dev)
    for step in range(3):
        data = _bytes(n, 100 + step)
        host_in.copy_(data)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(host_out, data + 1)


def test_copy_refuses_pageable_host_memory_and_overlap(cuda_lib):
    pa = cuda_lib
    lib = pa.load()
    pageable = np.zeros(4096, dtype=np.uint8)
    dev = torch.empty(4096, dtype=torch.uint8, device="cuda")
    p = pageable.ctypes.data
    p16 = p + (-p) % 16
    assert lib.pa_copy(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(p16), 1024, None) == \
        PA_ERR_INVALID_ARG
    assert lib.pa_copy(ctypes.c_void_p(dev.data_ptr() + 512), ctypes.c_void_p(dev.data_ptr()),
                       1024, None) == PA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        pa.copy(dev, torch.zeros(4096, dtype=torch.uint8))   # not pinned
