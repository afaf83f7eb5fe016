"""Pins of the oracle's bf16 / E8M0 / E4M3 codecs and its block quantizer.

Each check ties the oracle to something other than itself: hand-worked
blocks (tests/golden/hand_blocks.txt), exhaustive comparison with a library
conversion (torch's bf16 and float8_e4m3fn casts), a floating-point closed
form of the RCEIL exponent, and exact rational arithmetic.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from golden_io import hand_blocks


def f32_bits_to_bf16_torch(bits: np.ndarray) -> np.ndarray:
    f = torch.from_numpy(bits.view(np.float32).copy())
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
FINITE_BF16 = ALL_BF16[(ALL_BF16 & 0x7F80) != 0x7F80]


def test_bf16_round_matches_torch_on_random_and_tie_patterns():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=60000, dtype=np.uint64).astype(np.uint32)
    # exact ties (low half 0x8000) with odd and even upper halves, near-ties,
    # the overflow edge (largest bf16 and halfway to 2^128), subnormals
    up = rng.integers(0, 2**16, size=4000, dtype=np.uint64).astype(np.uint32)
    ties = (up << 16) | 0x8000
    near = np.concatenate([(up << 16) | 0x7FFF, (up << 16) | 0x8001])
    edge = np.array([0x7F7F0000, 0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0x7F7F8001,
                     0x00000001, 0x00008000, 0x00018000, 0x80008000, 0xFF7F8000], np.uint32)
    allb = np.concatenate([bits, ties, near, edge])
    f = allb.view(np.float32)
    keep = ~np.isnan(f)
    allb, f = allb[keep], f[keep]
    ours = np.array([O.bf16_round(float(x)) for x in f], np.uint16)
    ref = f32_bits_to_bf16_torch(allb)
    assert np.array_equal(ours, ref)


def test_bf16_roundtrip_exhaustive():
    lib = O.lib()
    for b in FINITE_BF16[::7]:
        v = lib.orc_bf16_to_double(int(b))
        assert lib.orc_bf16_round(v) == b


def _rceil_exact(a: Fraction) -> int:
    """Smallest integer e with a <= 448 * 2^e, by exact rational search."""
    e = 0
    while a > 448 * Fraction(2) ** e:
        e += 1
    while a <= 448 * Fraction(2) ** (e - 1):
        e -= 1
    return e


def test_e8m0_rceil_exhaustive_over_bf16_amax():
    pos = FINITE_BF16[(FINITE_BF16 & 0x8000) == 0]
    pos = pos[pos != 0]
    vals = bf16_to_f32(pos).astype(np.float64)
    for a in vals:
        b = O.e8m0_rceil(float(a))
        e = _rceil_exact(Fraction(float(a)))
        assert b == min(max(e, -127), 127) + 127, a
        # float closed form, away from the exact powers-of-two boundary
        r = a / 448.0
        if abs(math.log2(r) - round(math.log2(r))) > 1e-9:
            assert b == max(math.ceil(math.log2(r)), -127) + 127


@pytest.mark.parametrize("amax,byte", [(1.0, 119), (448.0, 127), (450.0, 128), (9984.0, 132),
                                       (256.0, 127), (2.0 ** -133, 0), (0.0, 0),
                                       (float("nan"), 255), (float("inf"), 255),
                                       (3.3895313892515355e38, 247)])
def test_e8m0_hand_values(amax, byte):
    assert O.e8m0_rceil(amax) == byte


SCALE_BYTES = [0, 1, 60, 100, 110, 119, 120, 126, 127, 128, 135, 150, 200, 247, 254]


def test_e4m3_encode_matches_torch_float8_for_all_bf16_and_scales():
    """y = x * 2^(127-b) for every finite bf16 x and a spread of scale bytes."""
    x = bf16_to_f32(FINITE_BF16).astype(np.float64)
    for b in SCALE_BYTES:
        y = np.ldexp(x, 127 - b)
        ok = np.abs(y) < 3.0e38               # stays inside fp32 for the torch cast
        ys = y[ok]
        ref = torch.from_numpy(np.clip(ys, -448.0, 448.0).astype(np.float32)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        ours = np.array([O.e4m3_encode(float(v)) for v in ys], np.uint8)
        assert np.array_equal(ours, ref), b


def test_e4m3_encode_brute_force_nearest_rational():
    """Nearest E4M3 value by exact rationals over all 126 finite magnitudes."""
    mags = [Fraction(O.e4m3_value(c)) for c in range(127)]
    rng = np.random.default_rng(1)
    ys = list(rng.uniform(-500, 500, 300)) + list(rng.uniform(-1, 1, 300) * 2.0 ** -6)
    ys += [m / 2 + mags[i + 1] / 2 for i, m in enumerate(mags[:-1])]   # every midpoint
    for y in ys:
        yf = Fraction(float(y))
        a = abs(yf)
        if a >= 448:
            want = 0x7E
        else:
            best = min(range(127), key=lambda c: (abs(mags[c] - a), c & 1))
            want = best
        want |= 0x80 if float(y) < 0 or (float(y) == 0 and math.copysign(1, float(y)) < 0) else 0
        assert O.e4m3_encode(float(y)) == want, y


def test_e4m3_specials():
    assert O.e4m3_encode(float("nan")) == 0x7F
    assert O.e4m3_encode(-0.0) == 0x80
    assert O.e4m3_encode(0.0) == 0x00
    assert O.e4m3_encode(-1e-9) == 0x80
    assert O.e4m3_encode(1e30) == 0x7E
    assert O.e4m3_encode(-float("inf")) == 0xFE
    assert O.e4m3_encode(464.0) == 0x7E      # above the last code, saturates
    assert O.e4m3_encode(2.0 ** -10) == 0x00  # tie to even (zero)


def _bf16_bits(v: float) -> int:
    b = f32_bits_to_bf16_torch(np.array([v], np.float32).view(np.uint32))[0]
    assert float(bf16_to_f32(np.array([b], np.uint16))[0]) == v or math.isnan(v)
    return int(b)


@pytest.mark.parametrize("case", list(hand_blocks()), ids=lambda c: c[0])
def test_hand_worked_blocks(case):
    name, vals, scale, codes = case
    bits = [_bf16_bits(v) for v in vals]
    s, q = O.quant_block(bits)
    assert s == scale, name
    assert list(q) == codes, name


def test_dequant_error_bound_and_max_code_on_random_blocks():
    """|x - q * 2^(b-127)| <= max(2^-4 |x|, 2^(b-127-10)); the block amax
    divided by the scale lies in (224, 448] (no clamp in play), so the
    largest code magnitude lies in [224, 448] after rounding."""
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(64, 32 * 16, generator=g) *
         torch.pow(2.0, torch.randint(-30, 30, (64, 1), generator=g).float())).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    out = O.quant_2d(xb, O.ROWWISE)
    xv = x.float().numpy().astype(np.float64)
    qv = torch.from_numpy(out["q_row"]).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    sc = out["s_row"].astype(np.int64) - 127
    scale = np.repeat(np.ldexp(1.0, sc), 32, axis=1)
    err = np.abs(xv - qv * scale)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, scale * 2.0 ** -10)
    assert np.all(err <= bound)
    blockmax = np.abs(qv).reshape(64, 16, 32).max(axis=2)
    assert np.all((blockmax >= 224) & (blockmax <= 448))
    amax = np.abs(xv).reshape(64, 16, 32).max(axis=2) / np.ldexp(1.0, sc)
    assert np.all((amax > 224) & (amax <= 448))
