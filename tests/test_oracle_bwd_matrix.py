"""Pins of the oracle's matrix backward (``swiglu_bwd_grads`` / ``swiglu_bwd``,
the loop over rows and columns that feeds the scalar gradient formulas).

Definition ("Add swiglu + MXFP8 fused CuTe DSL kernel", sections "API" and
"Numerics and tests"): the backward reads grad_h, gate and up, forms dGate
and dUp, rounds each to bf16 and casts them like the forward's activation.
The scalar formulas (``swiglu_grads_f64``, ``geglu_grads_f64``) are pinned
elsewhere by finite differences and hand-worked values; these tests pin the
matrix loop around them:

* every element of dgate / dup equals the pinned scalar result at the same
  (dh, gate, up), rounded fp32 -> bf16 by torch (not by the oracle), with dh
  strided differently from gate and up (ld_dh != ld_in) and gate, up the two
  halves of one packed buffer, for both activations;
* the hand-worked backward rows of tests/golden/swiglu_hand.txt come out of
  the matrix entry point;
* the matrix cast is the standalone quantizer of those gradients;
* the plausible slips -- operands passed in the wrong order, dh read with
  the gate/up row pitch -- give results these checks reject.
"""
import numpy as np
import pytest
import torch

import oracle as O
from golden_io import swiglu_hand

M, N = 37, 96                  # odd row count, three 32-column blocks
LD_IN = 2 * N + 16             # packed [gate | up | pad]
LD_DH = N + 40                 # dh rows sit in a wider buffer


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _inputs(seed):
    gen = torch.Generator().manual_seed(seed)
    packed = torch.zeros(M, LD_IN)
    packed[:, :N] = torch.randn(M, N, generator=gen) * 2.0          # gate
    packed[:, N:2 * N] = torch.randn(M, N, generator=gen) + 3.0     # up, shifted so a swap shows
    # rows to spare: the stride slip below reads M rows LD_IN elements apart
    dh_buf = torch.randn(2 * M, LD_DH, generator=gen) * 0.5 - 1.0
    pb, db = _bf16_bits(packed), _bf16_bits(dh_buf)
    return pb, db


def _views(pb, db):
    gate, up = pb[:, :N], pb[:, N:2 * N]
    dh = db[:M, 8:8 + N]
    assert gate.strides[0] // 2 == LD_IN and dh.strides[0] // 2 == LD_DH
    return dh, gate, up


def _value(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _expected(dh, gate, up, act):
    """Element by element: the scalar formula, fp32, then bf16 (torch RNE)."""
    scalar = O.geglu_grads_f64 if act == O.GELU else O.swiglu_grads_f64
    d, g, u = _value(dh), _value(gate), _value(up)
    dg = np.empty((M, N), np.float32)
    du = np.empty((M, N), np.float32)
    for r in range(M):
        for c in range(N):
            a, b = scalar(float(d[r, c]), float(g[r, c]), float(u[r, c]))
            dg[r, c], du[r, c] = np.float32(a), np.float32(b)
    return _bf16_bits(torch.from_numpy(dg)), _bf16_bits(torch.from_numpy(du))


@pytest.mark.parametrize("act", [O.SILU, O.GELU], ids=["silu", "gelu"])
def test_matrix_backward_is_the_scalar_formula_elementwise(act):
    pb, db = _inputs(21 + act)
    dh, gate, up = _views(pb, db)
    dg, du = O.swiglu_bwd_grads(dh, gate, up, act=act)
    want_dg, want_du = _expected(dh, gate, up, act)
    assert np.array_equal(dg, want_dg)
    assert np.array_equal(du, want_du)


@pytest.mark.parametrize("act", [O.SILU, O.GELU], ids=["silu", "gelu"])
def test_checks_reject_swapped_operands_and_a_wrong_dh_pitch(act):
    """What an argument slip in the matrix loop would return, computed through
    the same entry point with the operands permuted or dh re-strided: every
    one differs from the element-wise expectation in most elements."""
    pb, db = _inputs(31 + act)
    dh, gate, up = _views(pb, db)
    want_dg, want_du = _expected(dh, gate, up, act)
    # dh read with the gate/up row pitch: rows of dh_buf taken LD_IN apart
    flat = db.reshape(-1)
    assert 8 + (M - 1) * LD_IN + N <= flat.size
    dh_wrong_pitch = np.lib.stride_tricks.as_strided(flat[8:], shape=(M, N), strides=(2 * LD_IN, 2))
    slips = {
        "gate<->up": (dh, up, gate),
        "dh<->gate": (gate, dh, up),
        "dh<->up": (up, gate, dh),
        "dh pitch": (dh_wrong_pitch, gate, up),
    }
    for name, (a, b, c) in slips.items():
        dg, du = O.swiglu_bwd_grads(np.ascontiguousarray(a), np.ascontiguousarray(b), np.ascontiguousarray(c),
                                    act=act)
        wrong = (dg != want_dg).mean() + (du != want_du).mean()
        assert wrong > 0.5, (name, wrong)


def test_golden_backward_rows_through_the_matrix_entry_point():
    """One golden row per matrix row: gate and up in columns 0 and 2 of a
    4-wide buffer, dh in column 5 of a 7-wide one (different row pitches)."""
    rows = [r for r in swiglu_hand() if r[0] == "bwd"]
    k = len(rows)
    buf = torch.full((k, 4), 7.0)
    dhb = torch.full((k, 7), -5.0)
    for i, (_, dh, g, u, _, _) in enumerate(rows):
        buf[i, 0], buf[i, 2], dhb[i, 5] = g, u, dh
    pb, db = _bf16_bits(buf), _bf16_bits(dhb)
    dg, du = O.swiglu_bwd_grads(db[:, 5:6], pb[:, 0:1], pb[:, 2:3])
    for i, (_, _, _, _, want_dg, want_du) in enumerate(rows):
        assert _value(dg[i, 0]) == want_dg, (i, _value(dg[i, 0]), want_dg)
        assert _value(du[i, 0]) == want_du, (i, _value(du[i, 0]), want_du)


@pytest.mark.parametrize("act", [O.SILU, O.GELU], ids=["silu", "gelu"])
def test_matrix_backward_cast_is_the_standalone_quantizer_of_the_gradients(act):
    pb, db = _inputs(41 + act)
    gate, up = pb[:32, :N], pb[:32, N:2 * N]
    dh = db[:32, 8:8 + N]
    qg, qu, dg, du = O.swiglu_bwd(dh, gate, up, O.BOTH, act=act)
    for got, grads in ((qg, dg), (qu, du)):
        want = O.quant_2d(grads, O.BOTH)
        for key in want:
            assert np.array_equal(got[key], want[key]), key
