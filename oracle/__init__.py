"""CPU oracle for the MXFP8 cast path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library under
``mxfp8_quantization_moe_gb300``) never imports it, and the two share no
code, header, table or constant.

The arithmetic lives in ``mxfp8_oracle.c`` (plain C, IEEE double, no
contraction).  This module compiles it with gcc on first use, loads it with
ctypes and wraps it for numpy arrays.  Whole-matrix calls are split over row
ranges and run on a thread pool (ctypes releases the GIL), which changes
nothing in the arithmetic: every row is computed by the same plain loop.

Array conventions: bf16 tensors are ``np.uint16`` bit patterns; E4M3 codes
and E8M0 scale bytes are ``np.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROWWISE = 1
COLWISE = 2
BOTH = 3

SILU = 0      # activations of the gated forms
GELU = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i64, u8, u16, dbl = ctypes.c_int64, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_double
        vp = ctypes.c_void_p
        sig = {
            "orc_bf16_to_double": (dbl, [u16]),
            "orc_bf16_round": (u16, [ctypes.c_float]),
            "orc_bf16_from_double_via_fp32": (u16, [dbl]),
            "orc_e8m0_rceil": (u8, [dbl]),
            "orc_e4m3_to_double": (dbl, [u8]),
            "orc_e4m3_encode": (u8, [dbl]),
            "orc_quant_block": (None, [vp, i64, vp, i64, vp]),
            "orc_quant_2d": (None, [vp, i64, i64, i64, ctypes.c_int,
                                    vp, i64, vp, i64, vp, i64, vp, i64, i64, i64]),
            "orc_quant_3d_colwise": (None, [vp, i64, i64, i64, vp, vp, i64, i64]),
            "orc_sigmoid": (dbl, [dbl]),
            "orc_swiglu_h_f64": (dbl, [dbl, dbl]),
            "orc_swiglu_grads_f64": (None, [dbl, dbl, dbl, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]),
            "orc_swiglu_fwd": (None, [vp, vp, i64, i64, vp, i64, i64, i64]),
            "orc_swiglu_bwd": (None, [vp, i64, vp, vp, i64, i64, vp, vp, i64, i64, i64]),
            "orc_scales_blocked": (None, [vp, i64, i64, i64, i64, vp]),
            "orc_normal_cdf": (dbl, [dbl]),
            "orc_normal_pdf": (dbl, [dbl]),
            "orc_geglu_h_f64": (dbl, [dbl, dbl]),
            "orc_geglu_grads_f64": (None, [dbl, dbl, dbl, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]),
            "orc_gated_fwd": (None, [ctypes.c_int, vp, vp, i64, i64, vp, i64, i64, i64]),
            "orc_gated_bwd": (None, [ctypes.c_int, vp, i64, vp, vp, i64, i64, vp, vp, i64, i64, i64]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def lib():
    return _load()


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _split(lo: int, hi: int, parts: int, align: int):
    """Split [lo, hi) into up to ``parts`` ranges whose inner bounds are multiples of ``align``."""
    n_units = (hi - lo + align - 1) // align
    parts = max(1, min(parts, n_units))
    out = []
    for p in range(parts):
        a = lo + (n_units * p // parts) * align
        b = lo + (n_units * (p + 1) // parts) * align if p + 1 < parts else hi
        if b > a:
            out.append((a, min(b, hi)))
    return out


def _run_ranges(fn, lo, hi, threads, align):
    ranges = _split(lo, hi, threads, align)
    if len(ranges) <= 1:
        for a, b in ranges:
            fn(a, b)
        return
    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        list(ex.map(lambda ab: fn(*ab), ranges))


# ----------------------------------------------------------------- scalars

def bf16_round(f: float) -> int:
    return int(lib().orc_bf16_round(ctypes.c_float(f)))


def bf16_value(b: int) -> float:
    return float(lib().orc_bf16_to_double(b))


def e8m0_rceil(amax: float) -> int:
    return int(lib().orc_e8m0_rceil(amax))


def e4m3_encode(y: float) -> int:
    return int(lib().orc_e4m3_encode(y))


def e4m3_value(c: int) -> float:
    return float(lib().orc_e4m3_to_double(c))


def sigmoid(g: float) -> float:
    return float(lib().orc_sigmoid(g))


def normal_cdf(g: float) -> float:
    return _load().orc_normal_cdf(g)


def geglu_h_f64(g: float, u: float) -> float:
    return _load().orc_geglu_h_f64(g, u)


def geglu_grads_f64(dh: float, g: float, u: float):
    a, b = ctypes.c_double(), ctypes.c_double()
    _load().orc_geglu_grads_f64(dh, g, u, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def swiglu_h_f64(g: float, u: float) -> float:
    return float(lib().orc_swiglu_h_f64(g, u))


def swiglu_grads_f64(dh: float, g: float, u: float):
    a, b = ctypes.c_double(), ctypes.c_double()
    lib().orc_swiglu_grads_f64(dh, g, u, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def quant_block(v) -> tuple[int, np.ndarray]:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.uint16))
    assert v.shape == (32,)
    codes = np.zeros(32, np.uint8)
    scale = np.zeros(1, np.uint8)
    lib().orc_quant_block(_ptr(v), 1, _ptr(codes), 1, _ptr(scale))
    return int(scale[0]), codes


# ---------------------------------------------------------------- matrices

def quant_2d(x: np.ndarray, mode: int, rows=None, threads: int | None = None):
    """Quantize bf16 ``x`` (M, N) -> dict with q_row (M, N), s_row (M, N/32),
    q_col (N, M) [column-major data: q_col[c, r]], s_col (M/32, N).

    ``rows`` = (r_begin, r_end) restricts the work to those rows (colwise:
    whole 32-row blocks); outputs outside the range are left zero."""
    assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
    M, N = x.shape
    ldx = x.strides[0] // 2
    r0, r1 = (0, M) if rows is None else rows
    out = {}
    q_row = s_row = q_col = s_col = None
    if mode & ROWWISE:
        assert N % 32 == 0
        q_row = np.zeros((M, N), np.uint8)
        s_row = np.zeros((M, N // 32), np.uint8)
        out.update(q_row=q_row, s_row=s_row)
    if mode & COLWISE:
        assert M % 32 == 0 and r0 % 32 == 0 and r1 % 32 == 0
        q_col = np.zeros((N, M), np.uint8)
        s_col = np.zeros((M // 32, N), np.uint8)
        out.update(q_col=q_col, s_col=s_col)
    L = lib()

    def work(a, b):
        L.orc_quant_2d(_ptr(x), ldx, M, N, mode,
                       _ptr(q_row), N, _ptr(s_row), N // 32,
                       _ptr(q_col), M, _ptr(s_col), N, a, b)

    _run_ranges(work, r0, r1, threads or default_threads(), 32 if mode & COLWISE else 1)
    return out


def quant_3d_colwise(x: np.ndarray, experts=None, threads: int | None = None):
    """x: bf16 (E, N, K) contiguous -> q (E, K, N) [column-major per expert],
    s (E, N/32, K).  ``experts`` = (e_begin, e_end) restricts the work."""
    assert x.dtype == np.uint16 and x.ndim == 3 and x.flags.c_contiguous
    E, N, K = x.shape
    assert N % 32 == 0
    q = np.zeros((E, K, N), np.uint8)
    s = np.zeros((E, N // 32, K), np.uint8)
    e0, e1 = (0, E) if experts is None else experts
    L = lib()

    def work(a, b):
        L.orc_quant_3d_colwise(_ptr(x), E, N, K, _ptr(q), _ptr(s), a, b)

    _run_ranges(work, e0, e1, threads or default_threads(), 1)
    return q, s


def swiglu_fwd_h(gate: np.ndarray, up: np.ndarray, rows=None, threads: int | None = None, act: int = SILU):
    """bf16 h = bf16(fp32(act(gate) * up)) for (M, N) gate/up (same row stride);
    act = SILU (g sigma(g)) or GELU (g Phi(g))."""
    assert gate.dtype == np.uint16 and up.dtype == np.uint16 and gate.shape == up.shape
    assert gate.strides == up.strides and gate.strides[1] == 2
    M, N = gate.shape
    ld_in = gate.strides[0] // 2
    h = np.zeros((M, N), np.uint16)
    r0, r1 = (0, M) if rows is None else rows
    L = lib()

    def work(a, b):
        L.orc_gated_fwd(act, _ptr(gate), _ptr(up), ld_in, N, _ptr(h), N, a, b)

    _run_ranges(work, r0, r1, threads or default_threads(), 1)
    return h


def swiglu_bwd_grads(dh: np.ndarray, gate: np.ndarray, up: np.ndarray, rows=None,
                     threads: int | None = None, act: int = SILU):
    """bf16 (dgate, dup) for (M, N) inputs, activation ``act``."""
    assert gate.strides == up.strides and gate.strides[1] == 2 and dh.strides[1] == 2
    M, N = gate.shape
    ld_in = gate.strides[0] // 2
    ld_dh = dh.strides[0] // 2
    dg = np.zeros((M, N), np.uint16)
    du = np.zeros((M, N), np.uint16)
    r0, r1 = (0, M) if rows is None else rows
    L = lib()

    def work(a, b):
        L.orc_gated_bwd(act, _ptr(dh), ld_dh, _ptr(gate), _ptr(up), ld_in, N,
                        _ptr(dg), _ptr(du), N, a, b)

    _run_ranges(work, r0, r1, threads or default_threads(), 1)
    return dg, du


def swiglu_fwd(gate, up, mode, rows=None, threads=None, act=SILU):
    """Oracle of the fused forward: h, then the standalone 2D quantizer."""
    h = swiglu_fwd_h(gate, up, rows=rows, threads=threads, act=act)
    return quant_2d(h, mode, rows=rows, threads=threads), h


def swiglu_bwd(dh, gate, up, mode, rows=None, threads=None, act=SILU):
    """Oracle of the fused backward: dgate/dup, each through the 2D quantizer."""
    dg, du = swiglu_bwd_grads(dh, gate, up, rows=rows, threads=threads, act=act)
    return (quant_2d(dg, mode, rows=rows, threads=threads),
            quant_2d(du, mode, rows=rows, threads=threads), dg, du)


def scales_blocked(s: np.ndarray) -> np.ndarray:
    """An (R, C) uint8 scale matrix in the blocked 128 x 4 tile layout
    (zero-padded to multiples of 128 rows and 4 columns), flat.  For colwise
    scales pass the (N, M/32) view, i.e. the transpose of the (M/32, N)
    row-major scales."""
    R, C = s.shape
    rp, cp = -(-R // 128) * 128, -(-C // 4) * 4
    out = np.empty(rp * cp, np.uint8)
    st = s.strides
    base = s
    _load().orc_scales_blocked(base.ctypes.data, R, C, st[0], st[1], out.ctypes.data)
    return out


def _check_group_ends(ends, R: int, align: int) -> np.ndarray:
    ends = np.asarray(ends, np.int64)
    starts = np.concatenate([[0], ends[:-1]])
    assert ends.ndim == 1 and len(ends) >= 1 and ends[-1] == R
    assert np.all(ends >= starts)
    assert np.all(ends[:-1] % align == 0)
    return starts


def scales_blocked_m_groups(s: np.ndarray, group_end) -> np.ndarray:
    """Row scales of a tensor whose rows form consecutive groups (token
    groups of a grouped GEMM; ``group_end`` the cumulative end row of each
    group, the last = R), in the blocked layout with every group starting on
    a fresh 128-row tile: group g's rows go to padded rows starting at the
    sum of the earlier groups' sizes rounded up to 128 ("[mxfp8 moe
    training] add compile support": the M-groups scale swizzle and the upper
    bound rows + 128 * groups of the padded rows).  The padded matrix has
    (ceil(R/128) + G) * 128 rows (at least that bound) and the columns of
    ``scales_blocked``; it is zero outside the groups' rows.  Flat."""
    R, C = s.shape
    G = len(group_end)
    starts = _check_group_ends(group_end, R, 1)
    padded = np.zeros(((-(-R // 128) + G) * 128, C), np.uint8)
    o = 0
    for a, b in zip(starts, group_end):
        padded[o:o + (b - a)] = s[a:b]
        o += -(-(b - a) // 128) * 128
    return scales_blocked(padded)


def scales_blocked_k_groups(s: np.ndarray, group_end) -> np.ndarray:
    """Column scales, as the (N, M/32) matrix (the transpose of the (M/32, N)
    row-major scales), of a tensor whose M rows form consecutive groups
    (``group_end`` in rows of the tensor, multiples of 32 but the last = M):
    the blocked layout with every group's M/32-columns starting on a fresh
    4-column tile (the K-groups scale swizzle of the same page, upper bound
    cols + 4 * groups).  The padded matrix has N rows (as ``scales_blocked``
    pads them) and (ceil(M/128) + G) * 4 columns.  Flat."""
    N, C = s.shape
    G = len(group_end)
    M = int(group_end[-1])
    assert C == -(-M // 32)
    starts = _check_group_ends(group_end, M, 32)
    padded = np.zeros((N, (-(-M // 128) + G) * 4), np.uint8)
    o = 0
    for a, b in zip(starts, group_end):
        ca, cb = a // 32, -(-b // 32)
        padded[:, o:o + (cb - ca)] = s[:, ca:cb]
        o += -(-(cb - ca) // 4) * 4
    return scales_blocked(padded)


def scales_blocked_per_expert(s: np.ndarray) -> np.ndarray:
    """(E, R, C) scale matrices, one per expert, each in the blocked layout,
    one after another (the per-group 3D scale swizzle of "[mxfp8 moe
    training] add compile support").  Flat."""
    return np.concatenate([scales_blocked(np.ascontiguousarray(m)) for m in s])
