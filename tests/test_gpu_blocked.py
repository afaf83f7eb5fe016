"""Scales in the blocked layout (MXFP8_BLOCKED_SCALES) on the GPU.

* Parity: the kernels' blocked scale buffers equal the oracle's blocked
  transform of its plain scales (row scales as the (M, N/32) matrix, column
  scales as the (N, M/32) matrix), byte for byte including the zero padding,
  for the 2D quantizer and the fused forward and backward; data codes are
  unchanged by the flag.  Shapes leave partial 128-row and 4-column tiles.
* Pin of the layout itself: the oracle's blocked scales drive a block-scaled
  MXFP8 GEMM of the installed PyTorch (torch._scaled_mm with E8M0 scales);
  its result must match the product of the dequantised operands computed
  with the plain scales, and must stop matching when the oracle's layout is
  deliberately permuted.  Skipped where that GEMM is not available.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bits, compare_codes, u8
import mxfp8_quantization_moe_gb300 as mx

pytestmark = pytest.mark.gpu

B = mx.MXFP8_BLOCKED_SCALES
SHAPES = [(96, 160), (256, 512), (416, 4256)]


def _input(M, N, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((M, N), generator=g, device="cuda")
    x *= torch.pow(2.0, torch.randint(-20, 21, (M, 1), generator=g, device="cuda").float())
    x *= torch.pow(2.0, torch.randint(-6, 7, (1, N // 32), generator=g, device="cuda").float()).repeat_interleave(32, 1)
    return x.to(torch.bfloat16)


def _blocked_want(plain, mode):
    want = {}
    if mode & 1:
        want["s_row"] = O.scales_blocked(plain["s_row"])
    if mode & 2:
        want["s_col"] = O.scales_blocked(np.ascontiguousarray(plain["s_col"].T))
    return want


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_quant_2d_blocked_scales(shape, mode):
    M, N = shape
    x = _input(M, N, M + N)
    got = mx.quant_2d(x, mode | B)
    torch.cuda.synchronize()
    plain = O.quant_2d(bits(x), mode)
    want = _blocked_want(plain, mode)
    if mode & 1:
        assert np.array_equal(u8(got.q_row), plain["q_row"])
        assert np.array_equal(u8(got.s_row), want["s_row"])
    if mode & 2:
        assert np.array_equal(u8(got.q_col), plain["q_col"])
        assert np.array_equal(u8(got.s_col), want["s_col"])


@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_swiglu_fwd_blocked_scales(shape, mode):
    M, N = shape
    gate, up = _input(M, N, 7), _input(M, N, 8)
    got = mx.swiglu_fwd(gate, up, mode | B)
    torch.cuda.synchronize()
    plain, _ = O.swiglu_fwd(bits(gate), bits(up), mode)
    want = _blocked_want(plain, mode)
    for k, w in want.items():
        assert np.array_equal(u8(getattr(got, k)), w), k
    if mode & 1:
        compare_codes(u8(got.q_row), plain["q_row"], 1e-4, "q_row")
    if mode & 2:
        compare_codes(u8(got.q_col), plain["q_col"], 1e-4, "q_col")


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_swiglu_bwd_blocked_scales(mode):
    M, N = 256, 512
    dh, gate, up = _input(M, N, 11), _input(M, N, 12), _input(M, N, 13)
    got = mx.swiglu_bwd(dh, gate, up, mode | B)
    torch.cuda.synchronize()
    wg, wu, _, _ = O.swiglu_bwd(bits(dh), bits(gate), bits(up), mode)
    for h, plain in ((got.dgate(), wg), (got.dup(), wu)):
        want = _blocked_want(plain, mode)
        for k, w in want.items():
            assert np.array_equal(u8(getattr(h, k)), w), k
        if mode & 1:
            compare_codes(u8(h.q_row), plain["q_row"], 1e-4, "q_row")
        if mode & 2:
            compare_codes(u8(h.q_col), plain["q_col"], 1e-4, "q_col")


def _dequant_rows(q, s):
    v = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return v * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)


def _scaled_mm(qa, sa, qb, sb):
    A = torch.from_numpy(qa).cuda().view(torch.float8_e4m3fn)
    Bq = torch.from_numpy(qb).cuda().view(torch.float8_e4m3fn)
    SA = torch.from_numpy(sa).cuda().view(torch.float8_e8m0fnu)
    SB = torch.from_numpy(sb).cuda().view(torch.float8_e8m0fnu)
    return torch._scaled_mm(A, Bq.t(), scale_a=SA, scale_b=SB, out_dtype=torch.bfloat16).float().cpu().numpy()


def test_blocked_layout_drives_a_block_scaled_gemm():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this PyTorch has no E8M0 dtype")
    M, N, K = 256, 384, 512
    a, b = _input(M, K, 21), _input(N, K, 22)
    qa, qb = O.quant_2d(bits(a), O.ROWWISE), O.quant_2d(bits(b), O.ROWWISE)
    sa, sb = O.scales_blocked(qa["s_row"]), O.scales_blocked(qb["s_row"])
    try:
        got = _scaled_mm(qa["q_row"], sa, qb["q_row"], sb)
    except (RuntimeError, TypeError, ValueError, NotImplementedError) as e:
        pytest.skip("no block-scaled MXFP8 GEMM here: %s" % str(e).splitlines()[0])
    want = _dequant_rows(qa["q_row"], qa["s_row"]) @ _dequant_rows(qb["q_row"], qb["s_row"]).T
    scale = np.abs(_dequant_rows(qa["q_row"], qa["s_row"])).max(axis=1)[:, None] * \
        np.abs(_dequant_rows(qb["q_row"], qb["s_row"])).max(axis=1)[None, :] * K
    err = np.abs(got - want) / scale
    assert err.max() < 2.0 ** -9, err.max()
    # a wrong order inside the tiles must be caught: each tile's 512 bytes
    # taken as [4][32][4] instead of [32][4][4]
    bad = np.ascontiguousarray(sa.reshape(-1, 4, 32, 4).transpose(0, 2, 1, 3)).reshape(-1)
    wrong = _scaled_mm(qa["q_row"], bad, qb["q_row"], sb)
    assert (np.abs(wrong - want) / scale).max() > 2.0 ** -4


@pytest.mark.parametrize("mode", [1, 3])
def test_blocked_row_scales_at_a_4_byte_offset(mode):
    """Blocked row-scale buffers need only 4-byte alignment: scales at an
    offset of 4 bytes from a 16-byte boundary (the kernels' whole-chunk
    stores then step aside) must still equal the oracle's."""
    M, N = 256, 512
    gate, up = _input(M, N, 31), _input(M, N, 32)
    plain, _ = O.swiglu_fwd(bits(gate), bits(up), mode)
    nb = int(O.scales_blocked(plain["s_row"]).size)
    raw = torch.zeros(nb + 16, dtype=torch.uint8, device="cuda")
    s_row = raw[4:4 + nb]
    q_row = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    o = mx.MXFP8Cast(q_row=q_row, s_row=s_row)
    if mode & 2:
        o.q_col = torch.empty((N, M), dtype=torch.uint8, device="cuda")
        o.s_col = torch.zeros(int(O.scales_blocked(np.ascontiguousarray(plain["s_col"].T)).size),
                              dtype=torch.uint8, device="cuda")
    mx.swiglu_fwd(gate, up, mode | B, out=o)
    torch.cuda.synchronize()
    assert np.array_equal(u8(s_row), O.scales_blocked(plain["s_row"]))
    compare_codes(u8(q_row), plain["q_row"], 1e-4, "q_row")
