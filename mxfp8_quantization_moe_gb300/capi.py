"""ctypes binding of libmxfp8 (include/mxfp8.h), same names, argument marshalling only.

Every function takes raw device pointers (ints) and sizes exactly as the C
ABI does and returns the integer status; ``check`` turns a status into an
exception.  Loading fails loudly when the library has not been built -- there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmxfp8.so")

MXFP8_ROWWISE = 1
MXFP8_COLWISE = 2
MXFP8_BOTH = 3
MXFP8_BLOCKED_SCALES = 8   # flag: scales in the blocked 128 x 4 tile layout
ACT_SILU, ACT_GELU = 0, 1  # the gated activation of the *_grouped fused calls

STATUS_NAMES = {
    0: "MXFP8_OK", 1: "MXFP8_ERR_NULL", 2: "MXFP8_ERR_SHAPE", 3: "MXFP8_ERR_ALIGN",
    4: "MXFP8_ERR_LD", 5: "MXFP8_ERR_MODE", 6: "MXFP8_ERR_OVERLAP", 7: "MXFP8_ERR_LAUNCH",
    8: "MXFP8_ERR_DEVICE", 9: "MXFP8_ERR_CAPTURE",
}

# every symbol include/mxfp8.h declares, with (restype, argtypes)
_i64, _u64, _int, _vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "mxfp8_status_str": (ctypes.c_char_p, [_int]),
    "mxfp8_version": (_int, []),
    "mxfp8_init": (_int, [_vp]),
    "mxfp8_quant_2d": (_int, [_vp, _i64, _i64, _i64, _int,
                              _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "mxfp8_swiglu_fwd": (_int, [_vp, _vp, _i64, _i64, _i64, _int,
                                _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "mxfp8_swiglu_bwd": (_int, [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _int,
                                _vp, _vp, _i64, _vp, _vp, _i64,
                                _vp, _vp, _i64, _vp, _vp, _i64, _vp]),
    "mxfp8_quant_3d_colwise": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "mxfp8_device_status": (_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint64),
                                   _int, _vp]),
    "mxfp8_selftest_wait_timeout": (_int, [_u64, _vp]),
    "mxfp8_selftest_activation": (_int, [_vp, _vp]),
    "mxfp8_swiglu_fwd_noalloc": (_int, [_vp, _vp, _i64, _i64, _i64, _int,
                                        _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "mxfp8_swiglu_fwd_with_h": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp, _i64,
                                       _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "mxfp8_geglu_fwd": (_int, [_vp, _vp, _i64, _i64, _i64, _int,
                               _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "mxfp8_geglu_bwd": (_int, [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _int,
                               _vp, _vp, _i64, _vp, _vp, _i64,
                               _vp, _vp, _i64, _vp, _vp, _i64, _vp]),
    "mxfp8_selftest_activation_gelu": (_int, [_vp, _vp]),
    "mxfp8_quant_3d": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _vp, _vp, _vp, _vp]),
    "mxfp8_quant_2d_grouped": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _i64,
                                      _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "mxfp8_swiglu_fwd_grouped": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _i64,
                                        _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "mxfp8_swiglu_bwd_grouped": (_int, [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _i64,
                                        _vp, _vp, _i64, _vp, _vp,
                                        _vp, _vp, _i64, _vp, _vp, _vp]),
}


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__("%s%s" % (where + ": " if where else "", STATUS_NAMES.get(status, status)))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmxfp8.so is not built (%s); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def lib():
    return _lib


def check(status: int, where: str = "") -> None:
    if status != 0:
        raise MXFP8Error(status, where)


def mxfp8_status_str(s: int) -> str:
    return _lib.mxfp8_status_str(s).decode()


def mxfp8_version() -> int:
    return _lib.mxfp8_version()


def mxfp8_init(stream) -> int:
    return _lib.mxfp8_init(stream)


def mxfp8_quant_2d(x, ld_x, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                   q_col, ld_qcol, s_col, ld_scol, stream) -> int:
    return _lib.mxfp8_quant_2d(x, ld_x, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                               q_col, ld_qcol, s_col, ld_scol, stream)


def mxfp8_swiglu_fwd(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                     q_col, ld_qcol, s_col, ld_scol, stream) -> int:
    return _lib.mxfp8_swiglu_fwd(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                                 q_col, ld_qcol, s_col, ld_scol, stream)


def mxfp8_swiglu_bwd(dh, ld_dh, gate, up, ld_in, M, N, mode,
                     dg_row, du_row, ld_qrow, dg_srow, du_srow, ld_srow,
                     dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol, stream) -> int:
    return _lib.mxfp8_swiglu_bwd(dh, ld_dh, gate, up, ld_in, M, N, mode,
                                 dg_row, du_row, ld_qrow, dg_srow, du_srow, ld_srow,
                                 dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol, stream)


def mxfp8_quant_3d_colwise(x, E, N, K, q, s, stream) -> int:
    return _lib.mxfp8_quant_3d_colwise(x, E, N, K, q, s, stream)


def mxfp8_device_status(reset: bool, stream):
    """Returns (status, flags, fallbacks)."""
    f = ctypes.c_uint32(0)
    n = ctypes.c_uint64(0)
    st = _lib.mxfp8_device_status(ctypes.byref(f), ctypes.byref(n), 1 if reset else 0, stream)
    return st, int(f.value), int(n.value)


def mxfp8_selftest_wait_timeout(limit_cycles: int, stream) -> int:
    return _lib.mxfp8_selftest_wait_timeout(limit_cycles, stream)


def mxfp8_selftest_activation(out, stream) -> int:
    return _lib.mxfp8_selftest_activation(out, stream)


def mxfp8_swiglu_fwd_noalloc(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                             q_col, ld_qcol, s_col, ld_scol, stream) -> int:
    return _lib.mxfp8_swiglu_fwd_noalloc(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                                         q_col, ld_qcol, s_col, ld_scol, stream)


def mxfp8_swiglu_fwd_with_h(gate, up, ld_in, M, N, mode, h, ld_h, q_row, ld_qrow, s_row, ld_srow,
                            q_col, ld_qcol, s_col, ld_scol, stream) -> int:
    return _lib.mxfp8_swiglu_fwd_with_h(gate, up, ld_in, M, N, mode, h, ld_h, q_row, ld_qrow, s_row, ld_srow,
                                        q_col, ld_qcol, s_col, ld_scol, stream)


def mxfp8_geglu_fwd(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                    q_col, ld_qcol, s_col, ld_scol, stream) -> int:
    return _lib.mxfp8_geglu_fwd(gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow,
                                q_col, ld_qcol, s_col, ld_scol, stream)


def mxfp8_geglu_bwd(dh, ld_dh, gate, up, ld_in, M, N, mode,
                    dg_row, du_row, ld_qrow, dg_srow, du_srow, ld_srow,
                    dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol, stream) -> int:
    return _lib.mxfp8_geglu_bwd(dh, ld_dh, gate, up, ld_in, M, N, mode,
                                dg_row, du_row, ld_qrow, dg_srow, du_srow, ld_srow,
                                dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol, stream)


def mxfp8_selftest_activation_gelu(out, stream) -> int:
    return _lib.mxfp8_selftest_activation_gelu(out, stream)


def mxfp8_quant_3d(x, E, N, K, mode, q_row, s_row, q_col, s_col, stream) -> int:
    return _lib.mxfp8_quant_3d(x, E, N, K, mode, q_row, s_row, q_col, s_col, stream)


def mxfp8_quant_2d_grouped(x, ld_x, M, N, mode, group_end, num_groups, q_row, ld_qrow, s_row,
                           q_col, ld_qcol, s_col, stream) -> int:
    return _lib.mxfp8_quant_2d_grouped(x, ld_x, M, N, mode, group_end, num_groups, q_row, ld_qrow, s_row,
                                       q_col, ld_qcol, s_col, stream)


def mxfp8_swiglu_fwd_grouped(gate, up, ld_in, M, N, mode, act, group_end, num_groups,
                             q_row, ld_qrow, s_row, q_col, ld_qcol, s_col, stream) -> int:
    return _lib.mxfp8_swiglu_fwd_grouped(gate, up, ld_in, M, N, mode, act, group_end, num_groups,
                                         q_row, ld_qrow, s_row, q_col, ld_qcol, s_col, stream)


def mxfp8_swiglu_bwd_grouped(dh, ld_dh, gate, up, ld_in, M, N, mode, act, group_end, num_groups,
                             dg_row, du_row, ld_qrow, dg_srow, du_srow,
                             dg_col, du_col, ld_qcol, dg_scol, du_scol, stream) -> int:
    return _lib.mxfp8_swiglu_bwd_grouped(dh, ld_dh, gate, up, ld_in, M, N, mode, act, group_end, num_groups,
                                         dg_row, du_row, ld_qrow, dg_srow, du_srow,
                                         dg_col, du_col, ld_qcol, dg_scol, du_scol, stream)
