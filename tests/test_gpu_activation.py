"""Exhaustive check of the SwiGLU fast path's accuracy.

The fused kernels keep the fast fp32 activation (and gradient) values and
round them to bf16.  Their correctness argument rests on one fact: for every
bf16 gate value g in the fast range (g >= -64) the fast factors' relative
error is far below one bf16 step (2^-8), so a fast bf16 value is the
correctly rounded one or an adjacent bf16.  That caps every code difference
at one code and confines scale changes to blocks whose amax mantissa is 0x60
or 0x61, which the kernels recompute exactly.  The gate takes only 65536
values, so the fact is checked for all of them against the oracle's
double-precision sigmoid, with a wide margin (2^-12).
"""
import numpy as np
import pytest
import torch

import oracle as O
from mxfp8_quantization_moe_gb300 import capi, init

pytestmark = pytest.mark.gpu


def test_fast_path_error_is_far_below_one_bf16_step_for_every_gate():
    init()
    out = torch.empty(5 * 65536, dtype=torch.float32, device="cuda")
    assert capi.mxfp8_selftest_activation(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    v = out.view(5, 65536).cpu().numpy().astype(np.float64)
    g = (np.arange(65536, dtype=np.uint64) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    fast = np.isfinite(g) & (g >= -64.0)
    gf = g[fast]
    sig = np.array([O.sigmoid(float(x)) for x in gf])
    silu = gf * sig
    sn = 1.0 - sig
    big = gf > 20                       # 1 - sigma without cancellation for large g
    sn[big] = np.exp(-gf[big]) * sig[big]
    w = 1.0 + gf * sn
    dsilu = sig * w

    def rel(a, b):
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.abs(a - b) / np.abs(b)
        r[(a == b)] = 0.0
        return r

    u = 2.0 ** -24
    errs = {"sigma": rel(v[0][fast], sig) / u, "silu": rel(v[1][fast], silu) / u,
            "1-sigma": rel(v[2][fast], sn) / u, "silu'": rel(v[4][fast], dsilu) / u}
    print("max fast-path relative error (units of 2^-24): " +
          ", ".join("%s %.2f" % (k, e.max()) for k, e in errs.items()))
    for k, e in errs.items():
        assert np.all(np.isfinite(e)) and e.max() < 2.0 ** 12, (k, gf[np.argmax(e)])
