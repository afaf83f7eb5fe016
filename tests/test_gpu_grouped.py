"""Per-group blocked scales and the per-expert 3D quantizer on the GPU.

* mxfp8_quant_2d_grouped / mxfp8_swiglu_fwd_grouped / mxfp8_swiglu_bwd_grouped
  (both activations): data as the ungrouped oracle, row scales equal to the
  oracle's M-groups layout and column scales to its K-groups layout, byte for
  byte including the zero padding; group vectors with empty groups, groups
  smaller than a tile and a ragged last group (rowwise).
* invalid group ends: status bit 4, no scale written, data still written.
* the M-groups layout drives a block-scaled GEMM per group (torch._scaled_mm
  with E8M0 scales): each group's 128-row tiles are that group's scale operand.
* mxfp8_quant_3d: rowwise, colwise and both, plain and per-expert blocked
  scales, against the oracle (expert row count not a multiple of 128).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bits, compare_codes, u8
import mxfp8_quantization_moe_gb300 as mx
from mxfp8_quantization_moe_gb300 import capi, device_status

pytestmark = pytest.mark.gpu

CASES = [  # (M, N, group ends)
    (416, 160, [96, 96, 224, 416]),
    (1024, 288, [32, 160, 480, 992, 1024]),
    (640, 4256, [640]),
]


def _input(M, N, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((M, N), generator=g, device="cuda")
    x *= torch.pow(2.0, torch.randint(-12, 13, (M, 1), generator=g, device="cuda").float())
    return x.to(torch.bfloat16)


def _ends(e):
    return torch.tensor(e, dtype=torch.int32, device="cuda")


def _check(got, plain, ends, mode, what, exact=True):
    if mode & 1:
        assert np.array_equal(u8(got.s_row), O.scales_blocked_m_groups(plain["s_row"], ends)), what + " s_row"
        if exact:
            assert np.array_equal(u8(got.q_row), plain["q_row"]), what + " q_row"
        else:
            compare_codes(u8(got.q_row), plain["q_row"], 1e-4, what + " q_row")
    if mode & 2:
        want = O.scales_blocked_k_groups(np.ascontiguousarray(plain["s_col"].T), ends)
        assert np.array_equal(u8(got.s_col), want), what + " s_col"
        if exact:
            assert np.array_equal(u8(got.q_col), plain["q_col"]), what + " q_col"
        else:
            compare_codes(u8(got.q_col), plain["q_col"], 1e-4, what + " q_col")


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_quant_2d_grouped(case, mode):
    M, N, ends = CASES[case]
    x = _input(M, N, 100 + case)
    device_status(reset=True)
    got = mx.quant_2d_grouped(x, _ends(ends), mode)
    torch.cuda.synchronize()
    _check(got, O.quant_2d(bits(x), mode), ends, mode, "quant")
    assert device_status()[0] == 0


def test_quant_2d_grouped_ragged_rows_rowwise():
    M, N, ends = 400, 96, [64, 64, 320, 400]       # last group ends off a 32-row boundary
    x = _input(M, N, 7)
    got = mx.quant_2d_grouped(x, _ends(ends), 1)
    torch.cuda.synchronize()
    _check(got, O.quant_2d(bits(x), 1), ends, 1, "ragged")


@pytest.mark.parametrize("act", ["silu", "gelu"])
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_swiglu_fwd_bwd_grouped(act, mode):
    M, N, ends = 416, 160, [96, 96, 224, 416]
    gate, up, dh = _input(M, N, 1), _input(M, N, 2), _input(M, N, 3)
    a = O.SILU if act == "silu" else O.GELU
    got = mx.swiglu_fwd_grouped(gate, up, _ends(ends), mode, act=act)
    torch.cuda.synchronize()
    plain, _ = O.swiglu_fwd(bits(gate), bits(up), mode, act=a)
    _check(got, plain, ends, mode, "fwd", exact=False)
    g = mx.swiglu_bwd_grouped(dh, gate, up, _ends(ends), mode, act=act)
    torch.cuda.synchronize()
    wg, wu, _, _ = O.swiglu_bwd(bits(dh), bits(gate), bits(up), mode, act=a)
    _check(g.dgate(), wg, ends, mode, "dgate", exact=False)
    _check(g.dup(), wu, ends, mode, "dup", exact=False)
    assert device_status()[0] == 0


@pytest.mark.parametrize("ends", [[100, 416], [96, 64, 416], [96, 400]])
def test_invalid_group_ends_write_no_scales(ends):
    M, N = 416, 160
    x = _input(M, N, 5)
    device_status(reset=True)
    got = mx.quant_2d_grouped(x, _ends(ends), 3)
    flags, _ = device_status(reset=True)
    assert flags & 16
    assert not got.s_row.any() and not got.s_col.any()
    plain = O.quant_2d(bits(x), 3)
    assert np.array_equal(u8(got.q_row), plain["q_row"])
    assert np.array_equal(u8(got.q_col), plain["q_col"])


def test_m_groups_layout_drives_a_block_scaled_gemm_per_group():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this PyTorch has no E8M0 dtype")
    K, Nb = 256, 128
    ends = [128, 384, 512]                          # groups of 128, 256, 128 rows
    M = ends[-1]
    a = _input(M, K, 41)
    b = _input(Nb, K, 42)
    qa = mx.quant_2d_grouped(a, _ends(ends), 1)
    qb = mx.quant_2d(b, 1 | mx.MXFP8_BLOCKED_SCALES)
    torch.cuda.synchronize()
    tile = 128 * (-(-K // 128) * 4)                 # bytes of one 128-row tile row
    start, off = 0, 0
    for end in ends:
        n = end - start
        A = qa.q_row[start:end].view(torch.float8_e4m3fn)
        SA = qa.s_row[off:off + (n // 128) * tile].view(torch.float8_e8m0fnu)
        SB = qb.s_row.view(torch.float8_e8m0fnu)
        try:
            got = torch._scaled_mm(A, qb.q_row.view(torch.float8_e4m3fn).t(), scale_a=SA, scale_b=SB,
                                   out_dtype=torch.bfloat16).float()
        except (RuntimeError, TypeError, ValueError, NotImplementedError) as e:
            pytest.skip("no block-scaled MXFP8 GEMM here: %s" % str(e).splitlines()[0])
        want = a[start:end].float() @ b.float().t()
        rel = ((got - want).abs().max() / want.abs().max()).item()
        assert rel < 0.1, (start, rel)
        start, off = end, off + (n // 128) * tile


@pytest.mark.parametrize("blocked", [False, True])
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_quant_3d(mode, blocked):
    E, N, K = 3, 96, 160
    g = torch.Generator(device="cuda").manual_seed(9)
    x = (torch.randn((E, N, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    m = mode | (mx.MXFP8_BLOCKED_SCALES if blocked else 0)
    got = mx.quant_3d(x, m)
    torch.cuda.synchronize()
    xb = bits(x)
    if mode & 1:
        r = O.quant_2d(xb.reshape(E * N, K), O.ROWWISE)
        assert np.array_equal(u8(got.q_row).reshape(E * N, K), r["q_row"])
        s = r["s_row"].reshape(E, N, K // 32)
        want = O.scales_blocked_per_expert(s) if blocked else s
        assert np.array_equal(u8(got.s_row).reshape(-1), want.reshape(-1))
    if mode & 2:
        q, s = O.quant_3d_colwise(xb)
        assert np.array_equal(u8(got.q_col), q)
        want = O.scales_blocked_per_expert(np.ascontiguousarray(s.transpose(0, 2, 1))) if blocked else s
        assert np.array_equal(u8(got.s_col).reshape(-1), want.reshape(-1))
    assert device_status()[0] == 0
