"""The allocation-free forward (mxfp8_swiglu_fwd_noalloc), through the C ABI.

Some callers cannot allocate device memory themselves: code that must live
inside a host framework's fixed device-memory arena, or that runs where an
allocation would break the caller's rules (for example while it records
work it will replay).  This entry point gives them the forward with its
working memory -- the bf16 activation -- in scratch the library reserved
when it was loaded.  Every activation element takes the exactly rounded
path before the standalone cast, so the result must be the oracle's bit for
bit; against the fused forward (mxfp8_swiglu_fwd, whose fast activation is
within one bf16 step of the exact one) the scales are bit-exact and at most
1e-4 of the codes differ, by one code.  Both are checked on two calls in a
row: the second call reuses scratch that still holds the first call's
values.  A third case has a row length that is not a multiple of 8 (the
activation pass's element-by-element tail).

This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bits, compare_codes
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
    assert gate.stride() == up.stride()
    p = lambda k: o[k].data_ptr() if k in o else None
    ld = lambda k: o[k].stride(0) if k in o else 0
    return fn(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
              p("q_row"), ld("q_row"), p("s_row"), ld("s_row"),
              p("q_col"), ld("q_col"), p("s_col"), ld("s_col"),
              torch.cuda.current_stream().cuda_stream)


def _check(gate, up, mode, tag):
    """The allocation-free result against the oracle (bit-exact) and the
    fused forward (scales exact, codes within one)."""
    M, N = gate.shape
    want, got = _outs(M, N, mode), _outs(M, N, mode)
    assert _call(capi.mxfp8_swiglu_fwd, gate, up, mode, want) == 0
    assert _call(capi.mxfp8_swiglu_fwd_noalloc, gate, up, mode, got) == 0
    torch.cuda.synchronize()
    ref, _ = O.swiglu_fwd(bits(gate), bits(up), mode)
    for k in got:
        a, b = got[k].cpu().numpy(), want[k].cpu().numpy()
        assert np.array_equal(a, ref[k]), "%s %s: %d bytes differ from the oracle" % (tag, k, int((a != ref[k]).sum()))
        if k.startswith("s_"):
            assert np.array_equal(a, b), (tag, k)
        else:
            compare_codes(a, b, 1e-4, "%s %s" % (tag, k))


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_no_alloc_forward_equals_oracle_and_fused_forward_twice(mode):
    init()
    device_status(reset=True)
    shapes = [(1024, 4096), (2048, 2048 + 96)]     # the second call leaves stale scratch behind the first
    for call, (M, N) in enumerate(shapes):
        g = torch.Generator(device="cuda").manual_seed(1000 * mode + call)
        buf = torch.randn((M, 2 * N), generator=g, device="cuda")
        buf[:, :N] *= 2.0
        buf = buf.to(torch.bfloat16)
        _check(buf[:, :N], buf[:, N:], mode, "call %d" % call)   # packed [gate | up]
    flags, _ = device_status()
    assert flags == 0


def test_no_alloc_forward_ragged_row_length_colwise():
    """N = 100 (not a multiple of 8), row pitch 104: only the colwise cast
    accepts it; the activation pass handles the last 4 columns one by one."""
    init()
    device_status(reset=True)
    M, N, LD = 64, 100, 104
    g = torch.Generator(device="cuda").manual_seed(77)
    gbuf = (torch.randn((M, LD), generator=g, device="cuda") * 3.0).to(torch.bfloat16)
    ubuf = torch.randn((M, LD), generator=g, device="cuda").to(torch.bfloat16)
    for call in range(2):
        _check(gbuf[:, :N], ubuf[:, :N], 2, "ragged call %d" % call)
        gbuf, ubuf = ubuf * 2, gbuf
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
