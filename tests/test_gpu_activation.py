"""Exhaustive check of the SwiGLU fast path's rounding guard.

The fused kernels accept an fp32 activation value only if no bf16 rounding
boundary lies within a guard distance of it; otherwise they recompute it in
double.  Exactness therefore rests on one fact: for every bf16 gate value g in
the fast range (g >= -80), the fast factors' relative error, plus one
rounding for the final product and 1.5 ulps of margin, stays below the guard.
The gate takes only 65536 values, so the fact is checked for all of them,
against the oracle's double-precision sigmoid.
"""
import numpy as np
import pytest
import torch

import oracle as O
from mxfp8_quantization_moe_gb300 import capi, init

pytestmark = pytest.mark.gpu


def test_guard_bounds_fast_path_error_for_every_gate():
    init()
    out = torch.empty(8 * 65536, dtype=torch.float32, device="cuda")
    assert capi.mxfp8_selftest_activation(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    v = out.view(8, 65536).cpu().numpy().astype(np.float64)
    g = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    fast = np.isfinite(g) & (g >= -64.0)
    sig = np.array([O.sigmoid(float(x)) for x in g[fast]])
    gf = g[fast]
    silu = gf * sig
    sn = 1.0 - sig
    # 1 - sigma without cancellation for large g
    big = gf > 20
    sn[big] = np.exp(-gf[big]) * sig[big]
    w = 1.0 + gf * sn
    dsilu = sig * w

    def rel(a, b):
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.abs(a - b) / np.abs(b)
        r[(a == b)] = 0.0
        return r

    u = 2.0 ** -24
    e_s = rel(v[0][fast], sig) / u
    e_silu = rel(v[1][fast], silu) / u
    e_d = rel(v[4][fast], dsilu) / u
    # h = silu * u rounds once more; dup = (dh g) * sigma likewise
    need_h = e_silu + 1 + 1.5
    need_du = e_s + 1 + 1 + 1.5
    need_dg = e_d + 1 + 1 + 1.5
    print("max fast-path error (units of 2^-24): sigma %.3f silu %.3f silu' %.3f"
          % (e_s.max(), e_silu.max(), np.nanmax(e_d[np.isfinite(e_d)])))
    print("guard margins (ulps): h %.3f dup %.3f dgate %.3f"
          % ((v[5][fast] - need_h).min(), (v[6][fast] - need_du).min(),
             (v[7][fast] - need_dg).min()))
    # the dgate guard's shape: need_dg <= base + c * |w-1|/|w| -- report the
    # smallest c that works with the kernel's base
    wf = v[3][fast]
    fac = np.abs(wf - 1) / np.abs(wf)
    base = v[7][fast].min()
    big = fac > 0.05
    print("dgate: kernel base %.2f, needed cancel coefficient %.3f"
          % (base, np.max((need_dg[big] - base) / fac[big])))
    assert np.all(need_h <= v[5][fast]), gf[np.argmax(need_h - v[5][fast])]
    assert np.all(need_du <= v[6][fast]), gf[np.argmax(need_du - v[6][fast])]
    ok = need_dg <= v[7][fast]
    assert np.all(ok), gf[~ok][:10]
