"""GPU parity of the per-expert 3D colwise quantizer: bit-exact.

Small expert stacks (including N not a multiple of the tile height, so
tiles straddle experts) are compared whole, and so are the (E, 8192, 5120)
expert weights of the pages' benchmark table at every E it lists (1, 4, 16,
64), in the launch configuration the benchmark times (with 192-row tiles,
two of every three expert boundaries fall inside a tile).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import Guarded, bits, u8
import synthetic
from mxfp8_quantization_moe_gb300 import capi, device_status

pytestmark = pytest.mark.gpu


def run3d(x):
    E, N, K = x.shape
    q = Guarded((E, K, N))
    s = Guarded((E, N // 32, K))
    st = capi.mxfp8_quant_3d_colwise(x.data_ptr(), E, N, K, q.t.data_ptr(), s.t.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    assert q.intact() and s.intact()
    return q.t, s.t


@pytest.mark.parametrize("shape", [(1, 32, 64), (3, 96, 80), (2, 160, 136), (5, 64, 512), (4, 256, 72)],
                         ids=lambda s: "%dx%dx%d" % s)
def test_quant_3d_small_bit_exact(shape):
    E, N, K = shape
    g = torch.Generator(device="cuda").manual_seed(E * N + K)
    x = (torch.randn(shape, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x.view(-1)[::97] = float("nan") if E % 2 else 0.0
    q, s = run3d(x)
    wq, ws = O.quant_3d_colwise(bits(x).reshape(shape))
    assert np.array_equal(u8(q), wq)
    assert np.array_equal(u8(s), ws)


@pytest.mark.parametrize("E", [1, 4, 16, 64])
def test_quant_3d_experts_full(E):
    x = synthetic.experts(E, device="cuda")
    q, s = run3d(x)
    wq, ws = O.quant_3d_colwise(bits(x).reshape(x.shape))
    del x
    for e in range(E):
        assert np.array_equal(u8(q[e]), wq[e]), "expert %d data" % e
        assert np.array_equal(u8(s[e]), ws[e]), "expert %d scales" % e


def test_no_device_errors_after_3d():
    flags, _ = device_status()
    assert flags == 0
