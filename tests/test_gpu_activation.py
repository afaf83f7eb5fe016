"""Exhaustive check of the SwiGLU fast path's accuracy.

The fused kernels keep the fast fp32 activation (and gradient) values and
round them to bf16, recomputing exactly only the elements whose fast value
lies within a window around a 0x60/0x61 bf16 rounding midpoint (where a
scale byte could move).  The windows (64 fp32 ulps for h and dup, 512 for
dgate) are sized, with a margin of at least 2, from error bounds on the
gate-only factors: sigmoid and silu within 32 units of 2^-24, silu' within
256.  The gate takes only 65536 values, so those bounds are checked here for
all of them against the oracle's double-precision sigmoid, over the fast
range g >= -16.  Gates below -16 take the wide-range form, whose factor
2^120 e^g is checked the same way (within 8 units of 2^-24 wherever it is a
normal fp32 number, zero only where e^g is below 2^-246).
"""
import numpy as np
import pytest
import torch

import oracle as O
from mxfp8_quantization_moe_gb300 import capi, init

pytestmark = pytest.mark.gpu


def test_fast_path_error_bounds_for_every_gate():
    init()
    out = torch.empty(6 * 65536, dtype=torch.float32, device="cuda")
    assert capi.mxfp8_selftest_activation(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    v = out.view(6, 65536).cpu().numpy().astype(np.float64)
    g = (np.arange(65536, dtype=np.uint64) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    fast = np.isfinite(g) & (g >= -16.0)
    gf = g[fast]
    sig = np.array([O.sigmoid(float(x)) for x in gf])
    silu = gf * sig
    sn = 1.0 - sig
    big = gf > 20                       # 1 - sigma without cancellation for large g
    sn[big] = np.exp(-gf[big]) * sig[big]
    w = 1.0 + gf * sn
    dsilu = sig * w

    def rel(a, b):
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            r = np.abs(a - b) / np.abs(b)
        r[(a == b)] = 0.0
        return r

    u = 2.0 ** -24
    # the forward's silu comes scaled by 2^60: finite for every gate up to
    # 2^67 (beyond, it overflows to Inf, which the kernels recompute exactly)
    silu_up = v[1][fast] / 2.0 ** 60
    fin = np.abs(gf) < 2.0 ** 67
    assert np.all(np.isfinite(silu_up[fin]))
    assert np.all(np.isinf(silu_up[~fin]) | (rel(silu_up[~fin], silu[~fin]) <= 32 * 2.0 ** -24))
    # 1 - sigma is checked while it is a normal fp32 number with room to
    # spare; below 2^-100 the fast e^-g may flush to zero, harmlessly: there
    # g (1 - sigma) < 2^-90 vanishes against the 1 it is added to in silu'
    normal = sn >= 2.0 ** -100
    errs = {"sigma": (rel(v[0][fast], sig) / u, 32),
            "silu": (rel(silu_up[fin], silu[fin]) / u, 32),
            "1-sigma": (rel(v[2][fast][normal], sn[normal]) / u, 64),
            "silu'": (rel(v[4][fast], dsilu) / u, 256)}
    print("max fast-path relative error (units of 2^-24): " +
          ", ".join("%s %.2f" % (k, e.max()) for k, (e, _) in errs.items()))
    for k, (e, bound) in errs.items():
        assert np.all(np.isfinite(e)) and e.max() <= bound, (k, e.max(), bound)


def test_wide_range_factor_for_every_gate_below_the_fast_range():
    init()
    out = torch.empty(6 * 65536, dtype=torch.float32, device="cuda")
    assert capi.mxfp8_selftest_activation(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    v = out.view(6, 65536)[5].cpu().numpy().astype(np.float64)
    g = (np.arange(65536, dtype=np.uint64) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    far = np.isfinite(g) & (g < -16.0)
    gf, got = g[far], v[far]
    with np.errstate(under="ignore"):
        want = np.exp(gf) * 2.0 ** 120
    normal = want >= 2.0 ** -125
    rel = np.abs(got[normal] - want[normal]) / want[normal] / 2.0 ** -24
    print("wide-range factor: max relative error %.2f units of 2^-24 over %d gates" % (rel.max(), normal.sum()))
    assert rel.max() <= 8.0
    # below the normal range it may flush to zero, and only there: e^g < 2^-246
    small = ~normal
    assert np.all((got[small] == 0.0) | (np.abs(got[small] - want[small]) <= 2.0 ** -126))
    assert np.all(gf[got == 0.0] * np.log2(np.e) < -245.0)
