"""Pins of the oracle's GEGLU (h = gelu(g) * u, gelu(g) = g * Phi(g), the
exact erf form), independent of its own arithmetic:

* the forward for every bf16 gate against SciPy's normal CDF (its own
  implementation), rounded to fp32 then bf16;
* the backward closed form against central finite differences of a forward
  written here with CPython's own erfc;
* known values: Phi(1) = 0.841344746068543, Phi(0) = 1/2, gelu'(0) = 1/2,
  the limits for large |g|.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

scipy_special = pytest.importorskip("scipy.special")


def _bf16_of(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_forward_every_bf16_gate_against_scipy():
    g_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = (g_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ones = np.full(65536, 0x3F80, np.uint16)
    h = O.swiglu_fwd_h(g_bits[None, :].copy(), ones[None, :].copy(), act=O.GELU)[0]
    fin = np.isfinite(g) & (np.abs(g) < 1e30)
    ref = g[fin] * scipy_special.ndtr(g[fin])
    f32 = ref.astype(np.float32)
    # skip values whose double lies within 2^-40 of an fp32 rounding midpoint
    # (the two double evaluations may round to different fp32 there)
    with np.errstate(divide="ignore", invalid="ignore"):
        ulp = np.spacing(np.abs(f32)).astype(np.float64)
        frac = np.abs(ref) / ulp % 1.0
    ok = ~((np.abs(frac - 0.5) < 2.0 ** -14) & (ref != 0))
    want = _bf16_of(f32)
    got = h[fin]
    assert np.array_equal(got[ok], want[ok]), np.nonzero(got[ok] != want[ok])[0][:5]
    assert ok.sum() > 55000


def _h(g, u):
    return g * 0.5 * math.erfc(-g / math.sqrt(2.0)) * u


def test_backward_closed_form_matches_finite_differences():
    rng = np.random.default_rng(9)
    for _ in range(10000):
        g = float(rng.normal() * 3)
        u = float(rng.normal())
        dh = float(rng.normal())
        eps = 1e-5 * max(1.0, abs(g))
        fd_g = dh * (_h(g + eps, u) - _h(g - eps, u)) / (2 * eps)
        fd_u = dh * (_h(g, u + eps) - _h(g, u - eps)) / (2 * eps)
        dg, du = O.geglu_grads_f64(dh, g, u)
        assert abs(dg - fd_g) <= 1e-6 * (abs(dh * u) + 1e-300), (g, u, dh)
        assert abs(du - fd_u) <= 1e-6 * (abs(dh) * abs(g) + 1e-300), (g, u, dh)


def test_known_values_and_limits():
    assert O.normal_cdf(0.0) == 0.5
    assert abs(O.normal_cdf(1.0) - 0.841344746068543) < 1e-15
    assert abs(O.geglu_h_f64(1.0, 1.0) - 0.841344746068543) < 1e-15
    dg, du = O.geglu_grads_f64(1.0, 0.0, 1.0)
    assert dg == 0.5 and du == 0.0
    assert O.geglu_h_f64(40.0, 1.0) == 40.0                  # Phi = 1 to double precision
    assert O.geglu_h_f64(-40.0, 1.0) == 0.0 or abs(O.geglu_h_f64(-40.0, 1.0)) < 1e-300
    # far in the negative tail both gradients vanish
    dg, du = O.geglu_grads_f64(1.0, -40.0, 1.0)
    assert abs(dg) < 1e-300 and abs(du) < 1e-300
