"""GPU parity of the fused gated-activation kernels (SwiGLU and GEGLU) where
their fast arithmetic is weakest; same tolerance as the other SwiGLU tests
(scales bit-exact, codes within one, at most 1e-4 of them).

* rounding midpoints: every row block and column block holds one element
  whose exact fp32 value lies a few ulps from the bf16 rounding midpoint
  between mantissas 0x60 and 0x61 -- where the E8M0 RCEIL byte steps -- and
  that element is the block's amax;
* tiny gates (bf16 subnormals up to 2^-60) against huge ups / dh, so that
  g * sigmoid(g) is far below the normal fp32 range while the result is not;
* zero gates against non-finite ups, gates at the ends of the bf16 range.
The input values are picked with plain numpy / SciPy double arithmetic (only
to find candidates); the expected outputs come from the oracle.
"""
import numpy as np
import pytest
import torch
from scipy.special import ndtr

from test_gpu_swiglu import bwd_gpu, compare, fwd_gpu, oracle_bwd, oracle_fwd
from mxfp8_quantization_moe_gb300 import device_status

pytestmark = pytest.mark.gpu

MID = 0x608000          # fp32 mantissa field of the 0x60 | 0x61 bf16 midpoint
M = N = 256             # 8 x 8 tiles of 32 x 32


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)


def bf16(sign, exp, mant):
    """bf16 bit patterns from sign (0/1), unbiased exponent, 7-bit mantissa."""
    return ((np.asarray(sign, np.uint32) << 15) | ((np.asarray(exp, np.int64) + 127).astype(np.uint32) << 7)
            | np.asarray(mant, np.uint32)).astype(np.uint16)


def gates(lo=-64.0, hi=60.0, tiny=2.0 ** -20):
    b = np.arange(65536, dtype=np.uint32)
    g = (b << 16).view(np.float32).astype(np.float64)
    keep = np.isfinite(g) & (g >= lo) & (g <= hi) & (np.abs(g) >= tiny)
    return b[keep].astype(np.uint16), g[keep]


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def factors(act, g):
    """(activation f(g), its derivative f'(g), the gate band around the
    derivative's zero) for candidate search."""
    if act == "gelu":
        p = ndtr(g)
        return g * p, p + g * np.exp(-0.5 * g * g) / np.sqrt(2 * np.pi), (g > -1.0) & (g < -0.5)
    s = sigmoid(g)
    return g * s, s * (1 + g * (1 - s)), (g > -1.6) & (g < -1.0)


ACTS = ["silu", "gelu"]


def mid_dist(x):
    """Signed distance, in fp32 ulps, of fp32(x) from the 0x60|0x61 midpoint
    of its own binade."""
    f = np.abs(x).astype(np.float32).view(np.uint32).astype(np.int64)
    return (f & 0x7FFFFF) - MID


def hits_1d(factor, count=256):
    """The `count` pairs (gate index, mantissa k), over every gate and all
    128 mantissas, whose factor[g] * (1 + k/128) lies closest to a midpoint."""
    m = 1.0 + np.arange(128) / 128.0
    d = np.abs(mid_dist(factor[:, None] * m[None, :])).reshape(-1)
    best = np.argsort(d, kind="stable")[:count]
    return best // 128, best % 128


def diagonal_positions():
    """(row, col) of the element each 32x32 tile holds on its diagonal: every
    row block and every column block then holds exactly one."""
    r, c = [], []
    for bi in range(M // 32):
        for bj in range(N // 32):
            for t in range(32):
                r.append(32 * bi + t)
                c.append(32 * bj + t)
    return np.array(r), np.array(c)


def small_background(rng, scale_exp):
    """Gates in [-8, 8] and second operands below 2^scale_exp."""
    g = rng.uniform(-8, 8, (M, N)).astype(np.float32)
    x = (rng.uniform(-1, 1, (M, N)) * 2.0 ** scale_exp).astype(np.float32)
    return (torch.from_numpy(g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16),
            torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def fwd_midpoint_inputs(seed, act="silu"):
    gb, g = gates()
    f, _, _ = factors(act, g)
    gi, k = hits_1d(f)
    rng = np.random.default_rng(seed)
    gate, up = small_background(rng, -6)       # |h| < 8 * 2^-6 off the diagonal
    r, c = diagonal_positions()
    j = np.arange(len(r)) % len(gi)
    hv = f[gi[j]] * (1 + k[j] / 128.0)
    # exponent of up: the hit's |h| lands in [1, 2^20)
    e = rng.integers(0, 20, len(r)) - np.floor(np.log2(np.abs(hv))).astype(np.int64)
    gate[r, c] = gb[gi[j]]
    up[r, c] = bf16(rng.integers(0, 2, len(r)), e, k[j])
    return to_dev(gate), to_dev(up)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("seed", [0, 1])
def test_fwd_amax_at_rounding_midpoints(seed, act):
    gate, up = fwd_midpoint_inputs(seed, act)
    for mode in (1, 2, 3):
        compare(fwd_gpu(gate, up, mode, act=act), oracle_fwd(gate, up, mode, act=act), what="fwd-midpoint")


def bwd_midpoint_inputs(seed, which, act="silu"):
    rng = np.random.default_rng(seed)
    gb, g = gates()
    f, df, band = factors(act, g)
    if which == "dup":
        gi, k = hits_1d(f)                           # dup = dh * f(g)
        k2 = np.zeros_like(k)
    else:
        # dgate = (dh u) * f'(g): every gate against every pair of dh and u
        # mantissas; the closest 2048, plus the closest 256 among the gates
        # around the zero of f' (silu: g near -1.28, gelu: g near -0.75),
        # where f' is small and its fast value least accurate
        dsilu = df
        a = np.repeat(np.arange(128), 128)
        b = np.tile(np.arange(128), 128)
        prod = (1 + a / 128.0) * (1 + b / 128.0)
        picks = []
        for sel, count in ((np.arange(len(g)), 2048), (np.nonzero(band)[0], 256)):
            dist, idx = [], []
            for c0 in range(0, len(sel), 64):
                part = sel[c0:c0 + 64]
                d = np.abs(mid_dist(dsilu[part][:, None] * prod[None, :])).reshape(-1)
                keep = np.argpartition(d, count)[:count]
                dist.append(d[keep])
                idx.append(part[keep // len(prod)] * len(prod) + keep % len(prod))
            dist, idx = np.concatenate(dist), np.concatenate(idx)
            picks.append(idx[np.argsort(dist, kind="stable")[:count]])
        best = np.concatenate(picks)
        gi, pi = best // len(prod), best % len(prod)
        k, k2 = a[pi], b[pi]
    gate, up = small_background(rng, 1)
    _, dh = small_background(rng, -8)                # |dh u| < 2^-7 off the diagonal
    r, c = diagonal_positions()
    j = np.arange(len(r)) % len(gi)
    gate[r, c] = gb[gi[j]]
    if which == "dup":
        v = np.abs(f[gi[j]] * (1 + k[j] / 128.0))
        e = rng.integers(0, 20, len(r)) - np.floor(np.log2(v)).astype(np.int64)
        dh[r, c] = bf16(rng.integers(0, 2, len(r)), e, k[j])
        up[r, c] = bf16(0, -12, 0)                   # keeps dgate small there
    else:
        v = np.abs(df[gi[j]] * (1 + k[j] / 128.0) * (1 + k2[j] / 128.0))
        e = rng.integers(0, 20, len(r)) - np.floor(np.log2(v)).astype(np.int64)
        e1 = e // 2
        dh[r, c] = bf16(rng.integers(0, 2, len(r)), e1, k[j])
        up[r, c] = bf16(rng.integers(0, 2, len(r)), e - e1, k2[j])
    return to_dev(dh), to_dev(gate), to_dev(up)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("which", ["dgate", "dup"])
def test_bwd_amax_at_rounding_midpoints(which, act):
    dh, gate, up = bwd_midpoint_inputs(3, which, act)
    for mode in (1, 2, 3):
        dg, du = bwd_gpu(dh, gate, up, mode, act=act)
        wg, wu = oracle_bwd(dh, gate, up, mode, act=act)
        compare(dg, wg, what="dgate-midpoint(%s)" % which)
        compare(du, wu, what="dup-midpoint(%s)" % which)


def tiny_gate_inputs(seed):
    """Half the elements: |g| in [2^-133, 2^-60] (subnormal bf16 included)
    against |x| = 2^(-log2|g| + [-8, 8]); the rest ordinary values."""
    rng = np.random.default_rng(seed)
    n = M * N
    gexp = rng.integers(-133, -59, n)
    sub = gexp < -126
    # subnormal bf16: mantissa m in [64, 128) >> (-127 - e) is about 2^(e+133)
    gbits = np.where(sub,
                     (rng.integers(64, 128, n) >> np.clip(-127 - gexp, 0, 6)).astype(np.uint16),
                     bf16(0, np.maximum(gexp, -126), rng.integers(0, 128, n)))
    gbits = gbits | (rng.integers(0, 2, n).astype(np.uint16) << 15)
    gv = (gbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xexp = np.clip(-np.floor(np.log2(np.abs(gv))).astype(np.int64) + rng.integers(-8, 9, n), -126, 127)
    xbits = bf16(rng.integers(0, 2, n), xexp, rng.integers(0, 128, n))
    og = torch.from_numpy((rng.standard_normal(n) * 2).astype(np.float32)).to(torch.bfloat16)
    ox = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
    plain = rng.random(n) < 0.5
    gbits = np.where(plain, og.view(torch.int16).numpy().view(np.uint16), gbits)
    xbits = np.where(plain, ox.view(torch.int16).numpy().view(np.uint16), xbits)
    return gbits.reshape(M, N), xbits.reshape(M, N)


@pytest.mark.parametrize("act", ACTS)
def test_fwd_tiny_gates_huge_up(act):
    gbits, ubits = tiny_gate_inputs(5)
    gate, up = to_dev(gbits), to_dev(ubits)
    for mode in (1, 2, 3):
        compare(fwd_gpu(gate, up, mode, act=act), oracle_fwd(gate, up, mode, act=act), what="fwd-tiny-gate")


@pytest.mark.parametrize("act", ACTS)
def test_bwd_tiny_gates_huge_dh(act):
    gbits, dbits = tiny_gate_inputs(6)
    rng = np.random.default_rng(7)
    ubits = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    dh, gate, up = to_dev(dbits), to_dev(gbits), ubits.cuda()
    for mode in (1, 2, 3):
        dg, du = bwd_gpu(dh, gate, up, mode, act=act)
        wg, wu = oracle_bwd(dh, gate, up, mode, act=act)
        compare(dg, wg, what="dgate-tiny-gate")
        compare(du, wu, what="dup-tiny-gate")


@pytest.mark.parametrize("act", ACTS)
def test_special_values_mixed_in(act):
    """Zero gates against +-Inf / NaN ups (NaN blocks), gates at +-bf16 max
    and the smallest subnormal, a few gates below the fast range."""
    rng = np.random.default_rng(9)
    g = torch.from_numpy((rng.standard_normal((M, N)) * 2).astype(np.float32)).to(torch.bfloat16)
    u = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    dh = torch.from_numpy((rng.standard_normal((M, N)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    gv = g.view(torch.int16).numpy().view(np.uint16).copy()
    uv = u.view(torch.int16).numpy().view(np.uint16).copy()
    idx = rng.choice(M * N, 600, replace=False)
    # ... and both sides of -8 (the end of the GEGLU fast range)
    specials_g = np.array([0x0000, 0x8000, 0x7F7F, 0xFF7F, 0x0001, 0x8001, 0xC300, 0xC2FF, 0x42FF,
                           0xC100, 0xC101, 0xC0FF], np.uint16)
    specials_u = np.array([0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x7F7F, 0x3F80], np.uint16)
    gv.reshape(-1)[idx] = specials_g[np.arange(600) % len(specials_g)]
    uv.reshape(-1)[idx] = specials_u[(np.arange(600) // len(specials_g)) % len(specials_u)]
    gate, up, dhd = to_dev(gv), to_dev(uv), dh.cuda()
    for mode in (1, 2, 3):
        compare(fwd_gpu(gate, up, mode, act=act), oracle_fwd(gate, up, mode, act=act), what="fwd-specials")
        dg, du = bwd_gpu(dhd, gate, up, mode, act=act)
        wg, wu = oracle_bwd(dhd, gate, up, mode, act=act)
        compare(dg, wg, what="dgate-specials")
        compare(du, wu, what="dup-specials")
    flags, _ = device_status()
    assert flags == 0


@pytest.mark.parametrize("act", ACTS)
def test_both_mode_overflowing_fast_value_in_a_nan_row_block(act):
    """In "both" mode the column blocks are encoded from the row pass's
    settled values.  A row block holding a genuine NaN (a NaN up) and a
    value whose fast form overflows while the exact one is finite (the
    largest bf16 gate times up = 1: about 3.4e38) is a NaN block either way,
    but the finite value must still reach its column block exactly."""
    rng = np.random.default_rng(21)
    g = (rng.standard_normal((M, N)) * 2).astype(np.float32)
    u = rng.standard_normal((M, N)).astype(np.float32)
    dh = (rng.standard_normal((M, N)) * 0.05).astype(np.float32)
    to16 = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    gv, uv, dv = to16(g), to16(u), to16(dh)
    for k in range(8):
        r, c = 32 * k + 5, 32 * k + 7           # one per row block and column block
        gv[r, c], uv[r, c] = 0x7F7F, 0x3F80     # g = bf16 max, u = 1
        gv[r, c + 9], uv[r, c + 9] = 0x0000, 0x7FC0   # same row block: 0 * NaN
        dv[r, c] = 0x3F00                        # dh = 0.5
    gate, up, dhd = to_dev(gv), to_dev(uv), to_dev(dv)
    compare(fwd_gpu(gate, up, 3, act=act), oracle_fwd(gate, up, 3, act=act), what="fwd-both-overflow")
    dg, du = bwd_gpu(dhd, gate, up, 3, act=act)
    wg, wu = oracle_bwd(dhd, gate, up, 3, act=act)
    compare(dg, wg, what="dgate-both-overflow")
    compare(du, wu, what="dup-both-overflow")
    flags, _ = device_status()
    assert flags == 0
