"""The allocation-free forward (mxfp8_swiglu_fwd_noalloc) against the fused
forward (mxfp8_swiglu_fwd), through the C ABI.

The allocation-free entry point serves callers that cannot allocate device
memory themselves: it keeps the activation in scratch the library reserved
when it was loaded.  Its outputs must match the fused forward's within the
SwiGLU tolerance (scales bit-exact, at most 1e-4 of the codes one code
apart: the allocation-free path casts the exactly rounded activation, the
fused kernel a fast value within one bf16 step of it) on two calls in a row:
the second call reuses scratch that still holds the first call's values.
This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import numpy as np
import pytest
import torch

from gpu_util import compare_codes
from mxfp8_quantization_moe_gb300 import capi, device_status, init

pytestmark = pytest.mark.gpu

SCRATCH_ELEMS = 8 * 1024 * 1024


def _outs(M, N, mode):
    o = {}
    if mode & 1:
        o["q_row"] = torch.full((M, N), 0xA5, dtype=torch.uint8, device="cuda")
        o["s_row"] = torch.full((M, N // 32), 0xA5, dtype=torch.uint8, device="cuda")
    if mode & 2:
        o["q_col"] = torch.full((N, M), 0xA5, dtype=torch.uint8, device="cuda")
        o["s_col"] = torch.full((M // 32, N), 0xA5, dtype=torch.uint8, device="cuda")
    return o


def _call(fn, gate, up, mode, o):
    M, N = gate.shape
    p = lambda k: o[k].data_ptr() if k in o else None
    ld = lambda k: o[k].stride(0) if k in o else 0
    return fn(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
              p("q_row"), ld("q_row"), p("s_row"), ld("s_row"),
              p("q_col"), ld("q_col"), p("s_col"), ld("s_col"),
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_no_alloc_forward_equals_fused_forward_twice(mode):
    init()
    device_status(reset=True)
    shapes = [(1024, 4096), (2048, 2048 + 96)]     # the second call leaves stale scratch behind the first
    for call, (M, N) in enumerate(shapes):
        g = torch.Generator(device="cuda").manual_seed(1000 * mode + call)
        buf = torch.randn((M, 2 * N), generator=g, device="cuda")
        buf[:, :N] *= 2.0
        buf = buf.to(torch.bfloat16)
        gate, up = buf[:, :N], buf[:, N:]          # packed [gate | up]
        want, got = _outs(M, N, mode), _outs(M, N, mode)
        assert _call(capi.mxfp8_swiglu_fwd, gate, up, mode, want) == 0
        assert _call(capi.mxfp8_swiglu_fwd_noalloc, gate, up, mode, got) == 0
        torch.cuda.synchronize()
        for k in want:
            a, b = got[k].cpu().numpy(), want[k].cpu().numpy()
            if k.startswith("s_"):
                assert np.array_equal(a, b), (call, k)
            else:
                compare_codes(a, b, 1e-4, "call %d %s" % (call, k))
    flags, _ = device_status()
    assert flags == 0


def test_no_alloc_forward_rejects_problems_beyond_its_scratch():
    init()
    M, N = 4096, 4096                               # 16,777,216 elements > 8,388,608
    assert M * N > SCRATCH_ELEMS
    buf = torch.zeros((M, 2 * N), dtype=torch.bfloat16, device="cuda")
    o = _outs(M, N, 1)
    st = _call(capi.mxfp8_swiglu_fwd_noalloc, buf[:, :N], buf[:, N:], 1, o)
    assert st == 2, capi.STATUS_NAMES.get(st)       # MXFP8_ERR_SHAPE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((o["q_row"] == 0xA5).all())
