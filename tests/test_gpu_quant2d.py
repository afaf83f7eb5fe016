"""GPU parity of the standalone 2D quantizer against the oracle: bit-exact.

Shapes span several 128x64 tiles with ragged tails in both dimensions; the
data mixes per-row magnitudes over 2^-30..2^30 with NaN, Inf, zero blocks,
subnormals and E4M3-boundary values; one test runs every bf16 pattern.
Outputs sit in poisoned guard buffers that must come back untouched.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import Guarded, bits, u8
from mxfp8_quantization_moe_gb300 import capi, device_status

pytestmark = pytest.mark.gpu


def mixed_bf16(M, N, seed, ld=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    ld = ld or N
    x = torch.randn((M, ld), generator=g, device="cuda")
    x *= torch.pow(2.0, torch.randint(-30, 31, (M, 1), generator=g, device="cuda").float())
    x = x.to(torch.bfloat16)
    flat = x.view(-1)
    n = flat.numel()
    idx = torch.randint(0, n, (max(1, n // 2000),), generator=g, device="cuda")
    specials = torch.tensor([float("nan"), float("inf"), -float("inf"), 0.0, -0.0, 448.0, 450.0,
                             2.0 ** -133, -(2.0 ** -130), 9984.0], device="cuda").to(torch.bfloat16)
    flat[idx] = specials[torch.arange(idx.numel(), device="cuda") % specials.numel()]
    if M >= 32 and N >= 32:
        x[:32, :32] = 0                                # an all-zero block both ways
    return x[:, :N]


def run_quant(x, mode):
    M, N = x.shape
    outs = {}
    if mode & 1:
        outs["q_row"] = Guarded((M, N))
        outs["s_row"] = Guarded((M, N // 32))
    if mode & 2:
        outs["q_col"] = Guarded((N, M))
        outs["s_col"] = Guarded((M // 32, N))

    def p(k):
        return outs[k].t.data_ptr() if k in outs else None

    def ld(k):
        return outs[k].t.stride(0) if k in outs else 0

    st = capi.mxfp8_quant_2d(x.data_ptr(), x.stride(0), M, N, mode,
                             p("q_row"), ld("q_row"), p("s_row"), ld("s_row"),
                             p("q_col"), ld("q_col"), p("s_col"), ld("s_col"),
                             torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    for k, g in outs.items():
        assert g.intact(), "guard margin of %s overwritten" % k
    return {k: u8(g.t) for k, g in outs.items()}


SHAPES = [(32, 32), (128, 64), (160, 96), (256, 192), (96, 4096), (4096, 96), (1024, 1024)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_quant_2d_bit_exact(shape, mode):
    M, N = shape
    x = mixed_bf16(M, N, seed=M * 7 + N)
    got = run_quant(x, mode)
    want = O.quant_2d(bits(x), mode)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("shape,mode", [((100, 64), 1), ((33, 4096), 1), ((64, 40), 2), ((96, 200), 2)])
def test_quant_2d_ragged_free_dimension(shape, mode):
    """Rowwise needs only N % 32, colwise only M % 32: the other side is free."""
    M, N = shape
    x = mixed_bf16(M, N, seed=5)
    got = run_quant(x, mode)
    want = O.quant_2d(bits(x), mode)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_quant_2d_strided_input():
    x = mixed_bf16(256, 128, seed=9, ld=200)          # ld 200 elements (400 B, 16-aligned)
    assert x.stride(0) == 200
    got = run_quant(x, 3)
    want = O.quant_2d(bits(x), 3)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("shuffle", [False, True])
def test_quant_2d_every_bf16_pattern(shuffle):
    """All 65536 bf16 bit patterns, as (2048, 32) blocks and their transpose."""
    v = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if shuffle:
        v = np.random.default_rng(3).permutation(v)
    xb = v.reshape(2048, 32)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    got = run_quant(x, 1)
    want = O.quant_2d(xb, 1)
    for k in want:
        assert np.array_equal(got[k], want[k]), k
    xt = torch.from_numpy(np.ascontiguousarray(xb.T).view(np.int16)).cuda().view(torch.bfloat16)
    got = run_quant(xt, 2)
    want = O.quant_2d(np.ascontiguousarray(xb.T), 2)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_no_device_errors_after_quant():
    flags, _ = device_status()
    assert flags == 0


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_quant_2d_outputs_at_16_byte_strides(mode):
    """E4M3 outputs whose leading dimensions are 16 (not 32) modulo 32, so
    that every other 32-code block starts off a 32-byte boundary."""
    M, N = 160, 224
    x = mixed_bf16(M, N, seed=21)
    o = {}
    if mode & 1:
        o["q_row"] = Guarded((M, N + 16))
        o["s_row"] = Guarded((M, N // 32))
    if mode & 2:
        o["q_col"] = Guarded((N, M + 16))
        o["s_col"] = Guarded((M // 32, N))
    p = lambda k: o[k].t.data_ptr() if k in o else None
    ld = lambda k: o[k].t.stride(0) if k in o else 0
    st = capi.mxfp8_quant_2d(x.data_ptr(), x.stride(0), M, N, mode,
                             p("q_row"), ld("q_row"), p("s_row"), ld("s_row"),
                             p("q_col"), ld("q_col"), p("s_col"), ld("s_col"),
                             torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    want = O.quant_2d(bits(x), mode)
    for k, g in o.items():
        assert g.intact(), k
        got = u8(g.t)
        if k == "q_row":
            assert np.array_equal(got[:, :N], want[k])
            assert bool((got[:, N:] == 0xA5).all())
        elif k == "q_col":
            assert np.array_equal(got[:, :M], want[k])
            assert bool((got[:, M:] == 0xA5).all())
        else:
            assert np.array_equal(got, want[k]), k
