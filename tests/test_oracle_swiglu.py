"""Pins of the oracle's SwiGLU forward value and its backward closed form.

* hand-worked values (tests/golden/swiglu_hand.txt);
* the forward for every bf16 gate value against a 50-digit decimal
  evaluation of silu (independent arithmetic), rounded to fp32 then bf16;
* the backward closed form against central finite differences of an
  independent double-precision forward written here;
* limits and special cases (g = 0, large |g|, overflow to Inf).
"""
import math
import struct
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle as O
from golden_io import swiglu_hand


def bf16_of_float32(x: float) -> int:
    t = torch.tensor([x], dtype=torch.float32).to(torch.bfloat16)
    return int(t.view(torch.int16).item()) & 0xFFFF


def bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b << 16))[0]


@pytest.mark.parametrize("row", [r for r in swiglu_hand()], ids=lambda r: "%s%s" % (r[0], r[1:3]))
def test_hand_values(row):
    if row[0] == "fwd":
        _, g, u, h = row
        assert O.bf16_value(O.bf16_round(O.swiglu_h_f64(g, u))) == h
    else:
        _, dh, g, u, dg, du = row
        a, b = O.swiglu_grads_f64(dh, g, u)
        assert O.bf16_value(O.bf16_round(a)) == dg
        assert O.bf16_value(O.bf16_round(b)) == du


def _silu_decimal(g: float) -> Decimal:
    getcontext().prec = 50
    gd = Decimal(g)
    return gd / (1 + (-gd).exp())


def test_forward_every_bf16_gate_against_decimal_silu():
    """h(g, u=1) for all 65536 bf16 g: oracle vs a 50-digit decimal silu."""
    g_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = (g_bits.astype(np.uint32) << 16).view(np.float32)
    ones = np.full(65536, 0x3F80, np.uint16)
    h = O.swiglu_fwd_h(g_bits[None, :].copy(), ones[None, :].copy())[0]
    checked = 0
    for i in range(65536):
        gi = float(g[i])
        if math.isnan(gi):
            assert (h[i] & 0x7FFF) > 0x7F80
            continue
        if math.isinf(gi):
            want = 0x7F80 if gi > 0 else None       # silu(+inf) = +inf ; silu(-inf) = nan
            if want is None:
                assert (h[i] & 0x7FFF) > 0x7F80
            else:
                assert h[i] == want
            continue
        if gi < -1000.0:
            # g * e^g underflows far below fp32: -0 in fp32, -0 in bf16
            assert h[i] == 0x8000, gi
            continue
        if gi > 1000.0:
            assert h[i] == g_bits[i], gi             # sigma(g) = 1 to fp32 precision
            continue
        v = _silu_decimal(gi)
        f32 = np.float32(float(v))                  # decimal -> double -> fp32 (RN)
        # skip the (vanishingly rare) values within 2^-40 of an fp32 midpoint,
        # where the double step could round twice
        d = float(v)
        if d != 0.0:
            ulp = np.spacing(np.float32(abs(d)))
            frac = (abs(d) / float(ulp)) % 1.0
            if abs(frac - 0.5) < 2.0 ** -14:
                continue
        want = bf16_of_float32(float(f32))
        assert h[i] == want, (gi, float(v))
        checked += 1
    assert checked > 30000


def _h(g, u):
    return g / (1.0 + math.exp(-g)) * u


def test_backward_closed_form_matches_finite_differences():
    rng = np.random.default_rng(7)
    for _ in range(10000):
        g = float(rng.normal() * 3)
        u = float(rng.normal())
        dh = float(rng.normal())
        eps = 1e-5 * max(1.0, abs(g))
        fd_g = dh * (_h(g + eps, u) - _h(g - eps, u)) / (2 * eps)
        fd_u = dh * (_h(g, u + eps) - _h(g, u - eps)) / (2 * eps)
        dg, du = O.swiglu_grads_f64(dh, g, u)
        scale_g = abs(dh * u) + 1e-300
        scale_u = abs(dh) * (abs(g) + 1e-300)
        assert abs(dg - fd_g) <= 1e-6 * scale_g, (g, u, dh, dg, fd_g)
        assert abs(du - fd_u) <= 1e-6 * scale_u, (g, u, dh, du, fd_u)


def test_backward_special_points():
    dg, du = O.swiglu_grads_f64(2.0, 0.0, 3.0)
    assert dg == 0.5 * 2.0 * 3.0 and du == 0.0
    # large positive g: silu'(g) -> 1, silu(g) -> g
    dg, du = O.swiglu_grads_f64(1.0, 60.0, 1.0)
    assert dg == 1.0 and du == 60.0
    # large negative g: both vanish
    dg, du = O.swiglu_grads_f64(1.0, -800.0, 1.0)
    assert dg == 0.0 and du == 0.0


def test_forward_limits_and_overflow():
    assert O.swiglu_h_f64(0.0, 5.0) == 0.0
    assert O.swiglu_h_f64(80.0, 1.0) == 80.0
    assert abs(O.swiglu_h_f64(-30.0, 1.0)) < 1e-11
    # 3e38 * 3e38 overflows fp32: the bf16 result is +Inf and its block is a NaN block
    big = bits_to_float(0x7F61)
    hbits = O.bf16_round(O.swiglu_h_f64(big, big))
    assert hbits == 0x7F80
    blk = [hbits] + [0x3F80] * 31
    s, q = O.quant_block(blk)
    assert s == 255 and all(c == 0x7F for c in q)


def test_fused_forward_is_activation_then_standalone_quantizer():
    """The oracle's fused result is, by construction, quant_2d(h) -- checked here
    against a direct per-element evaluation of h with the scalar entry point."""
    gen = torch.Generator().manual_seed(11)
    buf = torch.randn(64, 128, generator=gen).to(torch.bfloat16)
    b = buf.view(torch.int16).numpy().view(np.uint16)
    gate, up = b[:, :64], b[:, 64:]
    out, h = O.swiglu_fwd(gate, up, O.BOTH)
    gf = buf[:, :64].double().numpy()
    uf = buf[:, 64:].double().numpy()
    for r in range(0, 64, 9):
        for c in range(0, 64, 5):
            assert h[r, c] == O.bf16_round(O.swiglu_h_f64(gf[r, c], uf[r, c]))
    q2 = O.quant_2d(h, O.BOTH)
    for k in q2:
        assert np.array_equal(q2[k], out[k])
