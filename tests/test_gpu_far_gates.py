"""GPU parity of the fused gated kernels for gates below the fast range.

SwiGLU gates below -16 take the wide-range evaluation (silu(g) = g e^g,
silu'(g) = (1 + g) e^g to a relative 2^-23, e^g formed with a 2^120 offset);
GEGLU gates below -6 (-8 in the backward but for per-group "both") take the
exact path.  Same tolerance as the other
gated tests (scales bit-exact, codes within one, at most 1e-4 of them):

* the block amax is a far-gate element whose exact value lies a few ulps
  from the 0x60|0x61 bf16 rounding midpoint (the scale byte steps there), in
  every row block and column block, forward and both backward outputs;
* far gates next to partners up to 2^121, where the wide-range factor
  flushes to zero while the true product is not negligible (those take the
  exact path), mixed with ordinary gates;
* the pages' mixed workload is compared whole in test_gpu_swiglu.py.
The inputs are picked with plain numpy double arithmetic (to find
candidates); the expected outputs come from the oracle.
"""
import numpy as np
import pytest
import torch

from test_gpu_swiglu import bwd_gpu, compare, fwd_gpu, oracle_bwd, oracle_fwd
from test_gpu_swiglu_edges import bf16, diagonal_positions, hits_1d, to_dev
from mxfp8_quantization_moe_gb300 import device_status

pytestmark = pytest.mark.gpu

M = N = 256


def far_gates(lo, hi):
    """bf16 patterns and values of the gates in [lo, hi]."""
    b = np.arange(65536, dtype=np.uint32)
    g = (b << 16).view(np.float32).astype(np.float64)
    keep = np.isfinite(g) & (g >= lo) & (g <= hi)
    return b[keep].astype(np.uint16), g[keep]


def bits_of(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def background(rng, exp):
    """Gates in [-8, 8], second operands below 2^exp (off the diagonal)."""
    g = bits_of(rng.uniform(-8, 8, (M, N)))
    x = bits_of(rng.uniform(-1, 1, (M, N)) * 2.0 ** exp)
    return g, x


def place(rng, factor, gb, low_exp, high_exp):
    """Diagonal (gate, operand) pairs whose product factor(g) * operand sits
    next to a 0x60|0x61 midpoint, with |product| in [2^low_exp, 2^high_exp)."""
    gi, k = hits_1d(factor)
    r, c = diagonal_positions()
    j = np.arange(len(r)) % len(gi)
    v = factor[gi[j]] * (1 + k[j] / 128.0)
    e = rng.integers(low_exp, high_exp, len(r)) - np.floor(np.log2(np.abs(v))).astype(np.int64)
    assert e.max() <= 127, "operand exponent beyond bf16"
    return r, c, gb[gi[j]], bf16(rng.integers(0, 2, len(r)), e, k[j])


def silu(g):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def dsilu(g):
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-g))
    return s * (1 + g * (1 - s))


@pytest.mark.parametrize("seed", [0, 1])
def test_fwd_far_gate_amax_at_rounding_midpoints(seed):
    gb, g = far_gates(-140.0, -16.1)
    rng = np.random.default_rng(seed)
    gate, up = background(rng, -118)
    r, c, gv, uv = place(rng, silu(g), gb, -100, -80)
    gate[r, c], up[r, c] = gv, uv
    gate, up = to_dev(gate), to_dev(up)
    for mode in (1, 2, 3):
        compare(fwd_gpu(gate, up, mode), oracle_fwd(gate, up, mode), what="fwd-far-midpoint")


@pytest.mark.parametrize("which", ["dgate", "dup"])
def test_bwd_far_gate_amax_at_rounding_midpoints(which):
    gb, g = far_gates(-140.0, -16.1)
    rng = np.random.default_rng(5 if which == "dgate" else 6)
    gate, dh = background(rng, -118)
    up = bits_of(rng.uniform(-1, 1, (M, N)))
    # dgate = dh * silu'(g) with u = +-1; dup = dh * silu(g)
    r, c, gv, dv = place(rng, dsilu(g) if which == "dgate" else silu(g), gb, -100, -80)
    gate[r, c], dh[r, c] = gv, dv
    if which == "dgate":
        up[r, c] = bf16(rng.integers(0, 2, len(r)), 0, 0)
    gate, up, dh = to_dev(gate), to_dev(up), to_dev(dh)
    for mode in (1, 2, 3):
        dg, du = bwd_gpu(dh, gate, up, mode)
        wg, wu = oracle_bwd(dh, gate, up, mode)
        compare(dg, wg, what="dgate-far-midpoint")
        compare(du, wu, what="dup-far-midpoint")


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_far_gates_next_to_huge_partners(act):
    """Half the gates in [-190, -16] (every one of them below the fast range)
    with partners up to 2^121, the rest ordinary; forward and backward in
    every mode."""
    rng = np.random.default_rng(11 if act == "silu" else 12)
    far = rng.random((M, N)) < 0.5
    g = np.where(far, -rng.uniform(16.1, 190, (M, N)), rng.uniform(-8, 8, (M, N)))
    ue = np.where(far, rng.integers(60, 122, (M, N)), rng.integers(-20, 40, (M, N)))
    u = rng.choice([-1.0, 1.0], (M, N)) * rng.uniform(1, 2, (M, N)) * 2.0 ** ue
    dh = rng.choice([-1.0, 1.0], (M, N)) * rng.uniform(1, 2, (M, N)) * 2.0 ** rng.integers(-20, 40, (M, N))
    gate, up, dh = to_dev(bits_of(g)), to_dev(bits_of(u)), to_dev(bits_of(dh))
    n = 0
    for mode in (1, 2, 3):
        n += compare(fwd_gpu(gate, up, mode, act=act), oracle_fwd(gate, up, mode, act=act), what="fwd-far-huge")
        dg, du = bwd_gpu(dh, gate, up, mode, act=act)
        wg, wu = oracle_bwd(dh, gate, up, mode, act=act)
        n += compare(dg, wg, what="dgate-far-huge") + compare(du, wu, what="dup-far-huge")
    print("differing codes:", n)




@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_far_gate_rows_of_every_density(act):
    """Rows whose share of gates below the fast range runs from none to all
    (row r of each 32-row block: share (r % 8) / 7), next to rows of isolated
    far gates: in a row pass the lanes then flag from 0 to all 16 pairs of
    their blocks, the case the warp settles cooperatively, with every count
    of flagged pairs across the lanes.  Forward and backward, every mode."""
    rng = np.random.default_rng(21 if act == "silu" else 22)
    share = (np.arange(M) % 8) / 7.0
    far = rng.random((M, N)) < share[:, None]
    far |= rng.random((M, N)) < 0.002
    g = np.where(far, -rng.uniform(16.1, 90, (M, N)), rng.normal(0.0, 2.0, (M, N)))
    u = rng.choice([-1.0, 1.0], (M, N)) * rng.uniform(1, 2, (M, N)) * 2.0 ** rng.integers(-10, 30, (M, N))
    dh = rng.normal(0.0, 1.0, (M, N))
    gate, up, dh = to_dev(bits_of(g)), to_dev(bits_of(u)), to_dev(bits_of(dh))
    n = 0
    for mode in (1, 2, 3):
        n += compare(fwd_gpu(gate, up, mode, act=act), oracle_fwd(gate, up, mode, act=act), what="fwd-far-rows")
        dg, du = bwd_gpu(dh, gate, up, mode, act=act)
        wg, wu = oracle_bwd(dh, gate, up, mode, act=act)
        n += compare(dg, wg, what="dgate-far-rows") + compare(du, wu, what="dup-far-rows")
    print("differing codes:", n)


def test_status_clean_after_far_gates():
    flags, _ = device_status()
    assert flags == 0
