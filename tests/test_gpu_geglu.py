"""GPU parity of the fused GEGLU forward and backward (the SwiGLU kernels with
the exact-erf GELU activation policy) against the oracle; same tolerance as
SwiGLU: scale bytes bit-exact, at most 1e-4 of the codes one code apart.
Also the exhaustive error bounds of the GEGLU fast path's gate-only factors,
which size its rounding-midpoint windows.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bits, u8
import synthetic
from mxfp8_quantization_moe_gb300 import capi, device_status, init
import mxfp8_quantization_moe_gb300 as mx
from test_gpu_swiglu import compare, rand_inputs

pytestmark = pytest.mark.gpu


def test_gelu_fast_path_error_bounds_for_every_gate():
    """Both fast paths: the tail table (forward, per-group backward "both"; fast range
    g >= -6) and the rational tail (the rest of the backward; g >= -8)."""
    init()
    out = torch.empty(5 * 65536, dtype=torch.float32, device="cuda")
    assert capi.mxfp8_selftest_activation_gelu(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    v = out.view(5, 65536).cpu().numpy().astype(np.float64)
    g = (np.arange(65536, dtype=np.uint64) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    sane = np.isfinite(g) & (np.abs(g) < 2.0 ** 100)
    p = np.full(65536, np.nan)
    d = np.full(65536, np.nan)
    p[sane] = [O.normal_cdf(float(x)) for x in g[sane]]
    d[sane] = [O.geglu_grads_f64(1.0, float(x), 1.0)[0] for x in g[sane]]

    def rel(a, b):
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.abs(a - b) / np.abs(b)
        r[(a == b)] = 0.0
        return r / 2.0 ** -24

    # the kernels' midpoint windows: 64, 64 and 512 fp32 ulps (table), 64 and
    # 1024 (rational tail); an error of e units of 2^-24 is e * 1.75 / 2 ulps
    # at the 0x60|0x61 midpoint mantissa, plus half an ulp for the multiply by
    # the exact product of inputs
    tab = sane & (g >= -6.0)
    poly = sane & (g >= -8.0)
    errs = {"Phi": (rel(v[0][tab], p[tab]), 16), "gelu": (rel(v[1][tab], g[tab] * p[tab]), 16),
            "gelu'": (rel(v[2][tab], d[tab]), 256),
            "Phi (rational)": (rel(v[3][poly], p[poly]), 32), "gelu' (rational)": (rel(v[4][poly], d[poly]), 768)}
    print("max GELU fast-path relative error (units of 2^-24): " +
          ", ".join("%s %.2f" % (k, e.max()) for k, (e, _) in errs.items()))
    for k, (e, bound) in errs.items():
        assert np.all(np.isfinite(e)) and e.max() <= bound, (k, e.max(), bound)


def oracle(gate, up, mode, dh=None):
    if dh is None:
        return O.swiglu_fwd(bits(gate), bits(up), mode, act=O.GELU)[0]
    r = O.swiglu_bwd(bits(dh), bits(gate), bits(up), mode, act=O.GELU)
    return r[0], r[1]


@pytest.mark.parametrize("shape", [(32, 64), (160, 96), (1024, 576)], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_geglu_fwd(shape, mode):
    gate, up, _ = rand_inputs(*shape, seed=shape[0] + mode)
    got = mx.swiglu_fwd(gate, up, mode, act="gelu")
    torch.cuda.synchronize()
    compare({k: u8(getattr(got, k)) for k in ("q_row", "s_row", "q_col", "s_col") if getattr(got, k) is not None},
            oracle(gate, up, mode), what="geglu fwd")


@pytest.mark.parametrize("shape", [(32, 64), (160, 96), (1024, 576)], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_geglu_bwd(shape, mode):
    gate, up, dh = rand_inputs(*shape, seed=shape[1] + mode)
    got = mx.swiglu_bwd(dh, gate, up, mode, act="gelu")
    torch.cuda.synchronize()
    wg, wu = oracle(gate, up, mode, dh)
    pick = lambda c: {k: u8(getattr(c, k)) for k in ("q_row", "s_row", "q_col", "s_col") if getattr(c, k) is not None}
    compare(pick(got.dgate()), wg, what="geglu dgate")
    compare(pick(got.dup()), wu, what="geglu dup")


def test_geglu_every_bf16_gate_and_mixed_workload():
    # every bf16 gate pattern (NaN/Inf included) against three up draws
    v = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    gate = torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
    g = torch.Generator(device="cuda").manual_seed(17)
    up = torch.randn((512, 128), generator=g, device="cuda").to(torch.bfloat16)
    dh = (torch.randn((512, 128), generator=g, device="cuda") * 0.1).to(torch.bfloat16)
    for mode in (1, 2, 3):
        got = mx.swiglu_fwd(gate, up, mode, act="gelu")
        gb = mx.swiglu_bwd(dh, gate, up, mode, act="gelu")
        torch.cuda.synchronize()
        compare({k: u8(getattr(got, k)) for k in ("q_row", "s_row", "q_col", "s_col") if getattr(got, k) is not None},
                oracle(gate, up, mode), what="geglu all-g fwd")
        wg, wu = oracle(gate, up, mode, dh)
        pick = lambda c: {k: u8(getattr(c, k)) for k in ("q_row", "s_row", "q_col", "s_col") if getattr(c, k) is not None}
        compare(pick(gb.dgate()), wg, what="geglu all-g dgate")
        compare(pick(gb.dup()), wu, what="geglu all-g dup")
    gate, up, dh = synthetic.mixed(device="cuda")
    got = mx.swiglu_fwd(gate, up, 3, act="gelu")
    gb = mx.swiglu_bwd(dh, gate, up, 3, act="gelu")
    torch.cuda.synchronize()
    n = compare({k: u8(getattr(got, k)) for k in ("q_row", "s_row", "q_col", "s_col")}, oracle(gate, up, 3),
                what="geglu mixed fwd")
    wg, wu = oracle(gate, up, 3, dh)
    pick = lambda c: {k: u8(getattr(c, k)) for k in ("q_row", "s_row", "q_col", "s_col")}
    n += compare(pick(gb.dgate()), wg, what="geglu mixed dgate") + compare(pick(gb.dup()), wu, what="geglu mixed dup")
    print("geglu mixed differing codes:", n)
    flags, _ = device_status()
    assert flags == 0
