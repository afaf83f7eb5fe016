"""Failure detection without a GPU fault: a wait nobody satisfies runs out its
(short) limit, the kernel records the error and returns, the host reads it,
and the context stays usable for the next launch."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bits, u8
from mxfp8_quantization_moe_gb300 import capi, device_status, init, quant_2d

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    init()
    device_status(reset=True)
    st = capi.mxfp8_selftest_wait_timeout(2_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    flags, _ = device_status(reset=True)
    assert flags & 8
    flags, _ = device_status()
    assert flags == 0
    # the context still works: a normal cast after the timed-out kernel
    x = torch.randn((64, 64), device="cuda").to(torch.bfloat16)
    o = quant_2d(x, 3)
    torch.cuda.synchronize()
    want = O.quant_2d(bits(x), 3)
    assert np.array_equal(u8(o.q_row), want["q_row"])
    assert np.array_equal(u8(o.q_col), want["q_col"])
    flags, _ = device_status()
    assert flags == 0


def test_status_before_graph_capture_and_capture_works():
    """After set-up, a cast can be captured in a CUDA graph and replayed."""
    init()
    x = torch.randn((256, 128), device="cuda").to(torch.bfloat16)
    out = quant_2d(x, 3)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        quant_2d(x, 3, out=out)
    x.copy_(torch.randn((256, 128), device="cuda").to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    want = O.quant_2d(bits(x), 3)
    assert np.array_equal(u8(out.q_row), want["q_row"])
    assert np.array_equal(u8(out.s_col), want["s_col"])
