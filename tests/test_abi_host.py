"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

* the library loads and exports every function include/mxfp8.h declares;
* every argument error returns its status code before the CUDA runtime is
  touched ("Add swiglu + MXFP8 fused CuTe DSL kernel", section "Numerics
  and tests": every launcher error path exercised), with fake pointers;
* calls that pass validation reach device set-up, which on a machine
  without a GPU reports MXFP8_ERR_DEVICE (only run where no GPU is present,
  since there the fake pointers would be launched on).
"""
import os
import re

import pytest
import torch

from mxfp8_quantization_moe_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULL, SHAPE, ALIGN, LD, MODE, OVERLAP, LAUNCH, DEVICE = range(9)
NO_GPU = not torch.cuda.is_available()

X = 0x10000000          # fake, 16-byte aligned "device" addresses, far apart
Q = 0x20000000
S = 0x30000000
QC = 0x40000000
SC = 0x50000000


def declared_functions():
    with open(os.path.join(ROOT, "include", "mxfp8.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mxfp8_swiglu_fwd", "mxfp8_swiglu_bwd", "mxfp8_quant_2d", "mxfp8_quant_3d_colwise"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = capi.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in capi.SIGNATURES, name


def test_status_strings_and_version():
    for s in range(10):
        assert capi.mxfp8_status_str(s).startswith("MXFP8_")
    assert capi.mxfp8_version() >= 100


def q2d(x=X, ld_x=256, M=128, N=256, mode=3, q_row=Q, ld_qrow=256, s_row=S, ld_srow=8,
        q_col=QC, ld_qcol=128, s_col=SC, ld_scol=256):
    return capi.mxfp8_quant_2d(x, ld_x, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                               q_col, ld_qcol, s_col, ld_scol, None)


@pytest.mark.parametrize("kw,status", [
    (dict(mode=0), MODE), (dict(mode=4), MODE), (dict(mode=-1), MODE),
    (dict(M=-1), SHAPE), (dict(N=-32), SHAPE),
    (dict(N=48, ld_x=48, ld_qrow=48, mode=1), SHAPE),          # rowwise needs N % 32
    (dict(M=100, mode=2), SHAPE),                                # colwise needs M % 32
    (dict(M=2 ** 31, mode=1), SHAPE),
    # more than 2^31 tiles of 96 x 128 (the kernels' 32-bit tile counters)
    (dict(M=2 ** 30, N=2 ** 16, ld_x=2 ** 16, ld_qrow=2 ** 16, ld_srow=2 ** 11, mode=1), SHAPE),
    (dict(x=0), NULL), (dict(q_row=0), NULL), (dict(s_row=0), NULL),
    (dict(q_col=0), NULL), (dict(s_col=0), NULL),
    (dict(x=X + 2), ALIGN), (dict(ld_x=260), ALIGN), (dict(q_row=Q + 8), ALIGN),
    (dict(ld_qrow=264), ALIGN), (dict(q_col=QC + 4), ALIGN), (dict(ld_qcol=136), ALIGN),
    (dict(ld_x=128), LD), (dict(ld_qrow=128), LD), (dict(ld_srow=4), LD),
    (dict(ld_qcol=96), LD), (dict(ld_scol=128), LD),
    (dict(q_row=X + 64), OVERLAP),                               # data over the input
    (dict(s_col=Q + 100), OVERLAP),                              # scales inside q_row
    (dict(q_col=Q + 4096), OVERLAP),                             # col data over row data
])
def test_quant_2d_argument_errors(kw, status):
    assert q2d(**kw) == status


def test_disabled_direction_pointers_are_ignored():
    # rowwise-only call with garbage colwise arguments still fails only on the
    # rowwise error it was given
    assert q2d(mode=1, q_col=3, s_col=0, ld_qcol=-5, ld_scol=-5, x=0) == NULL
    assert q2d(mode=2, q_row=3, s_row=0, ld_qrow=-5, ld_srow=-5, ld_x=260) == ALIGN


@pytest.mark.parametrize("kw", [dict(M=0), dict(N=0), dict(M=0, x=0, q_row=0)])
def test_empty_calls_succeed_without_device(kw):
    assert q2d(**kw) == OK


def _bwd_rowwise(du_off, base=0x20000000, sb=0x30000000, M=64, N=128):
    return capi.mxfp8_swiglu_bwd(X, N, X + 0x1000000, X + 0x1000000 + 2 * N, 2 * N, M, N, 1,
                                 base, base + du_off, 2 * N, sb, sb + N // 32, N // 16,
                                 None, None, 0, None, None, 0, None)


def test_overlap_check_is_exact_for_interleaved_layouts():
    N = 128
    # shifting dUp by 16 bytes into dGate's rows is an overlap
    assert _bwd_rowwise(N - 16) == OVERLAP
    # dUp's row end wrapping into the next dGate row
    assert _bwd_rowwise(N + 16) == OVERLAP


@pytest.mark.skipif(not NO_GPU, reason="would launch on fake pointers")
def test_interleaved_dgate_dup_halves_pass_validation():
    # rowwise outputs of two tensors interleaved in one buffer ([dGate | dUp])
    assert _bwd_rowwise(128) == DEVICE


@pytest.mark.skipif(not NO_GPU, reason="would launch on fake pointers")
def test_valid_calls_reach_device_setup():
    assert q2d() == DEVICE
    assert capi.mxfp8_init(None) == DEVICE
    # blocked scales ignore the scale leading dimensions
    assert q2d(mode=11, ld_srow=0, ld_scol=0) == DEVICE


def test_fwd_and_bwd_argument_errors():
    f = capi.mxfp8_swiglu_fwd
    assert f(X, 0, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == NULL
    assert f(X, X + 2, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == ALIGN
    assert f(X, X + 256, 200, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == LD
    assert f(X, X + 256, 512, 64, 256, 1, X + 1024, 256, S, 8, None, 0, None, 0, None) == OVERLAP
    b = capi.mxfp8_swiglu_bwd
    assert b(0, 256, X, X + 256, 512, 64, 256, 1, Q, Q + 256, 512, S, S + 8, 16,
             None, None, 0, None, None, 0, None) == NULL
    assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 1, Q, 0, 512, S, S + 8, 16,
             None, None, 0, None, None, 0, None) == NULL
    # [dGate | dUp] colwise halves, dUp shifted 16 bytes into dGate's last column
    assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 2, None, None, 0, None, None, 0,
             QC, QC + 256 * 64 - 16, 64, SC, SC + 256, 512, None) == OVERLAP
    if NO_GPU:   # valid packed layouts pass validation (fake pointers: never on a GPU)
        assert f(X, X + 256, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == DEVICE
        assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 2, None, None, 0, None, None, 0,
                 QC, QC + 256 * 64, 64, SC, SC + 256, 512, None) == DEVICE


def test_3d_argument_errors():
    f = capi.mxfp8_quant_3d_colwise
    assert f(X, 2, 48, 64, Q, S, None) == SHAPE           # N % 32
    assert f(X, 2, 64, 60, Q, S, None) == ALIGN           # K * 2 not a multiple of 16
    assert f(X, -1, 64, 64, Q, S, None) == SHAPE
    assert f(X, 0, 64, 64, Q, S, None) == OK              # empty
    assert f(0, 2, 64, 64, Q, S, None) == NULL
    assert f(X, 2, 64, 64, 0, S, None) == NULL
    assert f(X, 2, 64, 64, Q + 8, S, None) == ALIGN
    assert f(X, 2, 64, 64, X + 64, S, None) == OVERLAP    # data over the input
    assert f(X, 2 ** 19, 8192, 64, Q, S, None) == SHAPE    # E * N beyond the TMA coordinate range


def fwd_h(mode=1, h=0x60000000, ld_h=256, M=128, N=256, **kw):
    return capi.mxfp8_swiglu_fwd_with_h(X, X + 0x1000000, N, M, N, mode, h, ld_h,
                                        kw.get("q_row", Q), 256, S, 8, QC, 128, SC, 256, None)


@pytest.mark.parametrize("kw,status", [
    (dict(mode=2), MODE),                       # the activation comes from the row pass
    (dict(h=0), NULL),
    (dict(ld_h=128), LD),
    (dict(h=0x60000000 + 4), ALIGN), (dict(ld_h=260), ALIGN),
    (dict(h=Q + 256), OVERLAP),                 # h over the rowwise data
    (dict(h=X + 64), OVERLAP),                  # h over gate
])
def test_fwd_with_h_argument_errors(kw, status):
    assert fwd_h(**kw) == status


@pytest.mark.skipif(not NO_GPU, reason="would launch on fake pointers")
def test_fwd_with_h_valid_call_reaches_device_setup():
    assert fwd_h(mode=3) == DEVICE



def test_geglu_entry_points_validate_like_swiglu():
    f = capi.mxfp8_geglu_fwd
    assert f(X, 0, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == NULL
    assert f(X, X + 2, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == ALIGN
    assert f(X, X + 256, 200, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == LD
    assert f(X, X + 256, 512, 64, 256, 4, Q, 256, S, 8, None, 0, None, 0, None) == MODE
    assert f(X, X + 256, 512, 64, 256, 1, X + 1024, 256, S, 8, None, 0, None, 0, None) == OVERLAP
    assert f(X, X + 256, 512, 0, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == OK   # empty
    b = capi.mxfp8_geglu_bwd
    assert b(0, 256, X, X + 256, 512, 64, 256, 1, Q, Q + 256, 512, S, S + 8, 16,
             None, None, 0, None, None, 0, None) == NULL
    assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 2, None, None, 0, None, None, 0,
             QC, QC + 256 * 64 - 16, 64, SC, SC + 256, 512, None) == OVERLAP
    if NO_GPU:
        assert f(X, X + 256, 512, 64, 256, 1, Q, 256, S, 8, None, 0, None, 0, None) == DEVICE
        assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 2, None, None, 0, None, None, 0,
                 QC, QC + 256 * 64, 64, SC, SC + 256, 512, None) == DEVICE


def test_python_binding_rejects_unknown_activation():
    import mxfp8_quantization_moe_gb300 as mx
    g = torch.zeros((32, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mx.swiglu_fwd(g, g, 1, act="relu")
    with pytest.raises(ValueError):
        mx.swiglu_fwd(g, g, 1, act="gelu", keep_h=True)
    with pytest.raises(ValueError):
        mx.swiglu_bwd(g, g, g, 1, act="tanh")


GE = 0x70000000         # fake device address of a group-end vector


def q2d_grouped(M=128, N=256, mode=3, ge=GE, G=2, s_row=S, s_col=SC):
    return capi.mxfp8_quant_2d_grouped(X, N, M, N, mode, ge, G, Q, N, s_row, QC, M, s_col, None)


@pytest.mark.parametrize("kw,status", [
    (dict(ge=0), NULL),
    (dict(G=0), SHAPE), (dict(G=257), SHAPE),
    (dict(ge=GE + 2), ALIGN),
    (dict(mode=4), MODE),
    (dict(s_row=S + 2), ALIGN),                  # blocked row scales: 4-byte aligned
    (dict(ge=S + 64), OVERLAP),                  # group ends inside the row-scale buffer
    (dict(M=0), OK),                             # empty
])
def test_grouped_argument_errors(kw, status):
    assert q2d_grouped(**kw) == status


def test_grouped_scale_buffer_sizes_enter_the_overlap_check():
    # M = 128, N = 256, G = 2: row scales (1 + 2) * 128 rows * 8 bytes = 3072,
    # column scales 256 rows * (1 + 2) * 4 = 3072 bytes
    assert q2d_grouped(s_col=S + 3072 - 16) == OVERLAP
    if NO_GPU:
        assert q2d_grouped(s_col=S + 3072) == DEVICE


def test_grouped_fused_entry_points_check_the_activation():
    f = capi.mxfp8_swiglu_fwd_grouped
    assert f(X, X + 256, 512, 64, 256, 1, 2, GE, 1, Q, 256, S, None, 0, None, None) == MODE
    b = capi.mxfp8_swiglu_bwd_grouped
    assert b(X + 0x100000, 256, X, X + 256, 512, 64, 256, 1, 5, GE, 1, Q, Q + 256, 512, S, S + 4096,
             None, None, 0, None, None, None) == MODE
    if NO_GPU:
        assert f(X, X + 256, 512, 64, 256, 1, 1, GE, 1, Q, 256, S, None, 0, None, None) == DEVICE


def test_quant_3d_argument_errors():
    f = capi.mxfp8_quant_3d
    assert f(X, 2, 64, 64, 0, Q, S, QC, SC, None) == MODE
    assert f(X, 2, 64, 64, 16 | 1, Q, S, QC, SC, None) == MODE
    assert f(X, 2, 48, 64, 2, Q, S, QC, SC, None) == SHAPE           # colwise: N % 32
    assert f(X, 2, 48, 64, 1 | 8, Q, S, QC, SC, None) == SHAPE       # blocked: N % 32
    assert f(X, 2, 64, 48, 1, Q, S, QC, SC, None) == SHAPE           # rowwise: K % 32
    assert f(X, 2, 64, 60, 2, Q, S, QC, SC, None) == ALIGN           # K % 8
    assert f(X, 0, 64, 64, 3, Q, S, QC, SC, None) == OK
    assert f(X, 2, 64, 64, 1, 0, S, QC, SC, None) == NULL
    if NO_GPU:
        assert f(X, 2, 48, 64, 1, Q, S, QC, SC, None) == DEVICE      # rowwise plain: any N
