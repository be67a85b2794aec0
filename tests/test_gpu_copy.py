"""kvq_copy_async: pinned host <-> device copies by the SMs, also inside a captured CUDA graph."""

import ctypes

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq

pytestmark = pytest.mark.gpu


def test_pinned_and_device_round_trip():
    g = torch.Generator().manual_seed(5)
    host = torch.randint(0, 256, (458240,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.empty_like(host, device="cuda")
    kvq.kvq_copy(dev, host)
    back = torch.zeros_like(host).pin_memory()
    dev2 = torch.empty_like(dev)
    kvq.kvq_copy(dev2, dev)
    kvq.kvq_copy(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)
    assert torch.equal(back, host)


def test_inside_a_captured_step_with_new_host_contents():
    stream = torch.cuda.Stream()
    h_in = torch.zeros(4096, dtype=torch.float32).pin_memory()
    h_out = torch.zeros(4096, dtype=torch.float32).pin_memory()
    d = torch.zeros(4096, dtype=torch.float32, device="cuda")

    def fn():
        kvq.kvq_copy(d, h_in, stream=stream)
        with torch.cuda.stream(stream):
            d.mul_(2.0)
        kvq.kvq_copy(h_out, d, stream=stream)

    step = kvq.CapturedStep(fn, stream)
    for k in range(3):
        h_in.copy_(torch.arange(4096, dtype=torch.float32) + 100 * k)
        step()
        stream.synchronize()
        assert torch.equal(h_out, 2 * h_in)


def test_rejections_launch_nothing():
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ValueError):
        kvq.kvq_copy(dev, pageable)
    with pytest.raises(ValueError):
        kvq.kvq_copy(dev[:32], dev[32:48])
    lib = kvq.lib()
    buf = np.zeros(64, dtype=np.uint8)  # pageable host memory: refused by the C ABI's own check
    assert lib.kvq_copy_async(dev.data_ptr(), buf.ctypes.data, 64, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_copy_async(dev.data_ptr() + 8, dev.data_ptr() + 32, 16, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_copy_async(dev.data_ptr(), dev.data_ptr() + 16, 32, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_copy_async(dev.data_ptr(), dev.data_ptr() + 16, 24, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_copy_async(dev.data_ptr(), dev.data_ptr() + 16, 0, None) == kvq.KVQ_OK
    assert kvq.kvq_device_error() == (0, 0)
