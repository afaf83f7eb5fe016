"""mxfp8_quantization_moe_gb300 -- MXFP8 casts for MoE training on GB300.

The compute lives in ``libmxfp8.so`` (hand-written CUDA for sm_103a, C ABI in
``include/mxfp8.h``).  ``capi`` binds that ABI one-to-one; the helpers below
allocate outputs with PyTorch and call it.  Nothing here computes a cast on
the host: without the built library the import fails.

Layouts of the returned tensors (uint8):
  q_row (M, N) row-major,  s_row (M, N/32)
  q_col (N, M): q_col[c, r] is element (r, c) -- the column-major (M, N) data
  s_col (M/32, N)
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import capi
from .capi import MXFP8_BLOCKED_SCALES, MXFP8_BOTH, MXFP8_COLWISE, MXFP8_ROWWISE, MXFP8Error, check

__all__ = ["capi", "MXFP8Cast", "quant_2d", "swiglu_fwd", "swiglu_bwd", "quant_3d_colwise",
           "init", "device_status", "blocked_bytes", "MXFP8_ROWWISE", "MXFP8_COLWISE", "MXFP8_BOTH",
           "MXFP8_BLOCKED_SCALES", "MXFP8Error"]


@dataclass
class MXFP8Cast:
    q_row: Optional[torch.Tensor] = None
    s_row: Optional[torch.Tensor] = None
    q_col: Optional[torch.Tensor] = None
    s_col: Optional[torch.Tensor] = None
    h: Optional[torch.Tensor] = None      # the bf16 activation (forward with keep_h)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check_bf16_2d(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda:
        raise ValueError("%s must be a 2D bf16 CUDA tensor" % name)
    if t.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)


def blocked_bytes(rows: int, cols: int) -> int:
    """Bytes of a (rows, cols) scale matrix in the blocked layout (padded to
    multiples of 128 rows and 4 columns)."""
    return -(-rows // 128) * 128 * (-(-cols // 4) * 4)


def _alloc(M: int, N: int, mode: int, device, ld_row: Optional[int] = None) -> MXFP8Cast:
    """Outputs for one cast; with MXFP8_BLOCKED_SCALES the scale buffers are
    flat, zero-filled blocked matrices: (M, N/32) rowwise, (N, M/32) colwise."""
    out = MXFP8Cast()
    blocked = bool(mode & MXFP8_BLOCKED_SCALES)
    if mode & MXFP8_ROWWISE:
        out.q_row = torch.empty((M, N), dtype=torch.uint8, device=device)
        out.s_row = (torch.zeros(blocked_bytes(M, N // 32), dtype=torch.uint8, device=device) if blocked
                     else torch.empty((M, N // 32), dtype=torch.uint8, device=device))
    if mode & MXFP8_COLWISE:
        out.q_col = torch.empty((N, M), dtype=torch.uint8, device=device)
        out.s_col = (torch.zeros(blocked_bytes(N, M // 32), dtype=torch.uint8, device=device) if blocked
                     else torch.empty((M // 32, N), dtype=torch.uint8, device=device))
    return out


def _ld(t: Optional[torch.Tensor]) -> int:
    # flat (blocked) scale buffers have no leading dimension
    return t.stride(0) if t is not None and t.dim() == 2 else 0


def _lds(o: MXFP8Cast):
    return _ld(o.q_row), _ld(o.s_row), _ld(o.q_col), _ld(o.s_col)


def init(stream=None) -> None:
    check(capi.mxfp8_init(_stream(stream)), "mxfp8_init")


def quant_2d(x: torch.Tensor, mode: int = MXFP8_BOTH, out: Optional[MXFP8Cast] = None,
             stream=None) -> MXFP8Cast:
    """Standalone MXFP8 cast of a bf16 (M, N) tensor."""
    _check_bf16_2d(x, "x")
    M, N = x.shape
    o = out if out is not None else _alloc(M, N, mode, x.device)
    a, b, c, d = _lds(o)
    check(capi.mxfp8_quant_2d(x.data_ptr(), x.stride(0), M, N, mode,
                              _ptr(o.q_row), a, _ptr(o.s_row), b,
                              _ptr(o.q_col), c, _ptr(o.s_col), d, _stream(stream)), "mxfp8_quant_2d")
    return o


def swiglu_fwd(gate: torch.Tensor, up: Optional[torch.Tensor] = None, mode: int = MXFP8_BOTH,
               out: Optional[MXFP8Cast] = None, stream=None, keep_h: bool = False,
               act: str = "silu") -> MXFP8Cast:
    """Fused SwiGLU + MXFP8 cast.  With ``up=None``, ``gate`` is the packed
    [gate | up] (M, 2N) buffer.  With ``keep_h`` (rowwise modes) the bf16
    activation is returned too, in ``out.h``.  ``act="gelu"`` gives GEGLU."""
    if act not in ("silu", "gelu"):
        raise ValueError("act must be 'silu' or 'gelu'")
    if act == "gelu" and keep_h:
        raise ValueError("keep_h is available for SwiGLU only")
    if up is None:
        _check_bf16_2d(gate, "gate_up")
        n = gate.shape[1] // 2
        gate, up = gate[:, :n], gate[:, n:]
    _check_bf16_2d(gate, "gate")
    _check_bf16_2d(up, "up")
    if gate.shape != up.shape or gate.stride() != up.stride():
        raise ValueError("gate and up must have the same shape and strides")
    M, N = gate.shape
    o = out if out is not None else _alloc(M, N, mode, gate.device)
    a, b, c, d = _lds(o)
    if keep_h:
        if o.h is None:
            o.h = torch.empty((M, N), dtype=torch.bfloat16, device=gate.device)
        check(capi.mxfp8_swiglu_fwd_with_h(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
                                           o.h.data_ptr(), o.h.stride(0),
                                           _ptr(o.q_row), a, _ptr(o.s_row), b,
                                           _ptr(o.q_col), c, _ptr(o.s_col), d, _stream(stream)),
              "mxfp8_swiglu_fwd_with_h")
        return o
    fn = capi.mxfp8_geglu_fwd if act == "gelu" else capi.mxfp8_swiglu_fwd
    check(fn(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
             _ptr(o.q_row), a, _ptr(o.s_row), b,
             _ptr(o.q_col), c, _ptr(o.s_col), d, _stream(stream)), fn.__name__)
    return o


@dataclass
class SwiGLUGrads:
    """Packed [dGate | dUp] MXFP8 gradients.

    q_row (M, 2N), s_row (M, N/16); q_col (2N, M) column-major, s_col (M/32, 2N).
    With blocked scales, s_row and s_col are (2, bytes): one flat blocked
    matrix per gradient.
    """
    q_row: Optional[torch.Tensor] = None
    s_row: Optional[torch.Tensor] = None
    q_col: Optional[torch.Tensor] = None
    s_col: Optional[torch.Tensor] = None
    blocked: bool = False

    def dgate(self) -> MXFP8Cast:
        n = self._n()
        return MXFP8Cast(*self._halves(0, n))

    def dup(self) -> MXFP8Cast:
        n = self._n()
        return MXFP8Cast(*self._halves(1, n))

    def _n(self):
        return (self.q_row.shape[1] if self.q_row is not None else self.q_col.shape[0]) // 2

    def _halves(self, h, n):
        r = []
        r.append(None if self.q_row is None else self.q_row[:, h * n:(h + 1) * n])
        blocked = self.blocked
        if blocked:
            r.append(None if self.s_row is None else self.s_row[h])
        else:
            r.append(None if self.s_row is None else self.s_row[:, h * n // 32:(h + 1) * n // 32])
        r.append(None if self.q_col is None else self.q_col[h * n:(h + 1) * n])
        if blocked:
            r.append(None if self.s_col is None else self.s_col[h])
        else:
            r.append(None if self.s_col is None else self.s_col[:, h * n:(h + 1) * n])
        return r


def swiglu_bwd(dh: torch.Tensor, gate: torch.Tensor, up: Optional[torch.Tensor] = None,
               mode: int = MXFP8_BOTH, out: Optional[SwiGLUGrads] = None, stream=None,
               act: str = "silu") -> SwiGLUGrads:
    """Fused SwiGLU backward + MXFP8 cast of dgate and dup into packed
    [dGate | dUp] outputs.  With ``up=None``, ``gate`` is the packed input.
    ``act="gelu"`` gives the GEGLU backward."""
    if act not in ("silu", "gelu"):
        raise ValueError("act must be 'silu' or 'gelu'")
    if up is None:
        n = gate.shape[1] // 2
        gate, up = gate[:, :n], gate[:, n:]
    for t, nm in ((dh, "dh"), (gate, "gate"), (up, "up")):
        _check_bf16_2d(t, nm)
    if gate.shape != up.shape or gate.stride() != up.stride() or dh.shape != gate.shape:
        raise ValueError("dh, gate and up must have the same shape (gate/up the same strides)")
    M, N = gate.shape
    dev = gate.device
    blocked = bool(mode & MXFP8_BLOCKED_SCALES)
    o = out
    if o is None:
        o = SwiGLUGrads(blocked=blocked)
        if mode & MXFP8_ROWWISE:
            o.q_row = torch.empty((M, 2 * N), dtype=torch.uint8, device=dev)
            o.s_row = (torch.zeros((2, blocked_bytes(M, N // 32)), dtype=torch.uint8, device=dev) if blocked
                       else torch.empty((M, 2 * N // 32), dtype=torch.uint8, device=dev))
        if mode & MXFP8_COLWISE:
            o.q_col = torch.empty((2 * N, M), dtype=torch.uint8, device=dev)
            o.s_col = (torch.zeros((2, blocked_bytes(N, M // 32)), dtype=torch.uint8, device=dev) if blocked
                       else torch.empty((M // 32, 2 * N), dtype=torch.uint8, device=dev))
    qr = o.q_row.data_ptr() if o.q_row is not None else None
    sr = o.s_row.data_ptr() if o.s_row is not None else None
    qc = o.q_col.data_ptr() if o.q_col is not None else None
    sc = o.s_col.data_ptr() if o.s_col is not None else None
    ld_qrow = o.q_row.stride(0) if o.q_row is not None else 0
    ld_qcol = o.q_col.stride(0) if o.q_col is not None else 0
    if blocked:
        # one flat blocked matrix per gradient
        sr2 = None if sr is None else o.s_row[1].data_ptr()
        sc2 = None if sc is None else o.s_col[1].data_ptr()
        ld_srow = ld_scol = 0
    else:
        ld_srow = o.s_row.stride(0) if o.s_row is not None else 0
        ld_scol = o.s_col.stride(0) if o.s_col is not None else 0
        sr2 = None if sr is None else sr + N // 32
        sc2 = None if sc is None else sc + N
    fn = capi.mxfp8_geglu_bwd if act == "gelu" else capi.mxfp8_swiglu_bwd
    check(fn(
        dh.data_ptr(), dh.stride(0), gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
        qr, None if qr is None else qr + N, ld_qrow,
        sr, sr2, ld_srow,
        qc, None if qc is None else qc + N * ld_qcol, ld_qcol,
        sc, sc2, ld_scol,
        _stream(stream)), fn.__name__)
    return o


def quant_3d_colwise(x: torch.Tensor, q: Optional[torch.Tensor] = None,
                     s: Optional[torch.Tensor] = None, stream=None):
    """(E, N, K) bf16 -> q (E, K, N) uint8 [per-expert column-major data],
    s (E, N/32, K) uint8 scales."""
    if x.dtype != torch.bfloat16 or x.dim() != 3 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous (E, N, K) bf16 CUDA tensor")
    E, N, K = x.shape
    if q is None:
        q = torch.empty((E, K, N), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((E, N // 32, K), dtype=torch.uint8, device=x.device)
    check(capi.mxfp8_quant_3d_colwise(x.data_ptr(), E, N, K, q.data_ptr(), s.data_ptr(),
                                      _stream(stream)), "mxfp8_quant_3d_colwise")
    return q, s


def grouped_scale_bytes(M: int, N: int, num_groups: int):
    """(row-scale bytes, column-scale bytes) of one cast with per-group
    blocked scales (M-groups rows, K-groups columns) for M rows in
    ``num_groups`` token groups."""
    t = -(-M // 128) + num_groups
    return t * 128 * (-(-N // 128) * 4), -(-N // 128) * 128 * t * 4


def _groups(group_end: torch.Tensor):
    if group_end.dtype != torch.int32 or group_end.dim() != 1 or not group_end.is_contiguous():
        raise ValueError("group_end must be a contiguous 1-D int32 tensor of cumulative end rows")
    return group_end.data_ptr(), group_end.numel()


def _act_id(act: str) -> int:
    if act not in ("silu", "gelu"):
        raise ValueError("act must be 'silu' or 'gelu'")
    return capi.ACT_GELU if act == "gelu" else capi.ACT_SILU


def _alloc_grouped(M, N, mode, G, device, n_out=1):
    rb, cb = grouped_scale_bytes(M, N, G)
    shape = (lambda b: (n_out, b)) if n_out > 1 else (lambda b: (b,))
    o = {}
    if mode & MXFP8_ROWWISE:
        o["q_row"] = torch.empty((M, n_out * N), dtype=torch.uint8, device=device)
        o["s_row"] = torch.zeros(shape(rb), dtype=torch.uint8, device=device)
    if mode & MXFP8_COLWISE:
        o["q_col"] = torch.empty((n_out * N, M), dtype=torch.uint8, device=device)
        o["s_col"] = torch.zeros(shape(cb), dtype=torch.uint8, device=device)
    return o


def quant_2d_grouped(x: torch.Tensor, group_end: torch.Tensor, mode: int = MXFP8_BOTH,
                     out: Optional[MXFP8Cast] = None, stream=None) -> MXFP8Cast:
    """MXFP8 cast of a bf16 (M, N) tensor whose rows form token groups
    (``group_end``: int32 device tensor of cumulative end rows), scales in the
    per-group blocked layouts (flat, zero-filled buffers)."""
    _check_bf16_2d(x, "x")
    M, N = x.shape
    gp, G = _groups(group_end)
    o = out if out is not None else MXFP8Cast(**_alloc_grouped(M, N, mode, G, x.device))
    check(capi.mxfp8_quant_2d_grouped(x.data_ptr(), x.stride(0), M, N, mode, gp, G,
                                      _ptr(o.q_row), _ld(o.q_row), _ptr(o.s_row),
                                      _ptr(o.q_col), _ld(o.q_col), _ptr(o.s_col), _stream(stream)),
          "mxfp8_quant_2d_grouped")
    return o


def swiglu_fwd_grouped(gate: torch.Tensor, up: torch.Tensor, group_end: torch.Tensor,
                       mode: int = MXFP8_BOTH, act: str = "silu", out: Optional[MXFP8Cast] = None,
                       stream=None) -> MXFP8Cast:
    """Fused gated activation + MXFP8 cast with per-group blocked scales."""
    _check_bf16_2d(gate, "gate")
    _check_bf16_2d(up, "up")
    if gate.shape != up.shape or gate.stride() != up.stride():
        raise ValueError("gate and up must have the same shape and strides")
    M, N = gate.shape
    gp, G = _groups(group_end)
    o = out if out is not None else MXFP8Cast(**_alloc_grouped(M, N, mode, G, gate.device))
    check(capi.mxfp8_swiglu_fwd_grouped(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
                                        _act_id(act), gp, G, _ptr(o.q_row), _ld(o.q_row), _ptr(o.s_row),
                                        _ptr(o.q_col), _ld(o.q_col), _ptr(o.s_col), _stream(stream)),
          "mxfp8_swiglu_fwd_grouped")
    return o


def swiglu_bwd_grouped(dh: torch.Tensor, gate: torch.Tensor, up: torch.Tensor, group_end: torch.Tensor,
                       mode: int = MXFP8_BOTH, act: str = "silu", out: Optional[SwiGLUGrads] = None,
                       stream=None) -> SwiGLUGrads:
    """Fused gated-activation backward + MXFP8 cast into packed [dGate | dUp]
    data, one per-group blocked scale buffer per gradient."""
    for t, nm in ((dh, "dh"), (gate, "gate"), (up, "up")):
        _check_bf16_2d(t, nm)
    if gate.shape != up.shape or gate.stride() != up.stride() or dh.shape != gate.shape:
        raise ValueError("dh, gate and up must have the same shape (gate/up the same strides)")
    M, N = gate.shape
    gp, G = _groups(group_end)
    o = out if out is not None else SwiGLUGrads(blocked=True, **_alloc_grouped(M, N, mode, G, gate.device, n_out=2))
    qr = _ptr(o.q_row)
    qc = _ptr(o.q_col)
    ld_qcol = _ld(o.q_col)
    check(capi.mxfp8_swiglu_bwd_grouped(
        dh.data_ptr(), dh.stride(0), gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
        _act_id(act), gp, G,
        qr, None if qr is None else qr + N, _ld(o.q_row),
        _ptr(None if o.s_row is None else o.s_row[0]), _ptr(None if o.s_row is None else o.s_row[1]),
        qc, None if qc is None else qc + N * ld_qcol, ld_qcol,
        _ptr(None if o.s_col is None else o.s_col[0]), _ptr(None if o.s_col is None else o.s_col[1]),
        _stream(stream)), "mxfp8_swiglu_bwd_grouped")
    return o


def quant_3d(x: torch.Tensor, mode: int = MXFP8_BOTH, out: Optional[MXFP8Cast] = None,
             stream=None) -> MXFP8Cast:
    """(E, N, K) bf16 expert weights -> rowwise q_row (E, N, K) + s_row
    (E, N, K/32) and/or colwise q_col (E, K, N) [per-expert column-major] +
    s_col (E, N/32, K); with MXFP8_BLOCKED_SCALES each expert's scales as one
    blocked matrix, flat per expert: s_row (E, bytes), s_col (E, bytes)."""
    if x.dtype != torch.bfloat16 or x.dim() != 3 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous (E, N, K) bf16 CUDA tensor")
    E, N, K = x.shape
    blocked = bool(mode & MXFP8_BLOCKED_SCALES)
    if out is not None:
        check(capi.mxfp8_quant_3d(x.data_ptr(), E, N, K, mode, _ptr(out.q_row), _ptr(out.s_row),
                                  _ptr(out.q_col), _ptr(out.s_col), _stream(stream)), "mxfp8_quant_3d")
        return out
    o = MXFP8Cast()
    dev = x.device
    if mode & MXFP8_ROWWISE:
        o.q_row = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
        o.s_row = (torch.zeros((E, blocked_bytes(N, K // 32)), dtype=torch.uint8, device=dev) if blocked
                   else torch.empty((E, N, K // 32), dtype=torch.uint8, device=dev))
    if mode & MXFP8_COLWISE:
        o.q_col = torch.empty((E, K, N), dtype=torch.uint8, device=dev)
        o.s_col = (torch.zeros((E, blocked_bytes(K, N // 32)), dtype=torch.uint8, device=dev) if blocked
                   else torch.empty((E, N // 32, K), dtype=torch.uint8, device=dev))
    check(capi.mxfp8_quant_3d(x.data_ptr(), E, N, K, mode, _ptr(o.q_row), _ptr(o.s_row),
                              _ptr(o.q_col), _ptr(o.s_col), _stream(stream)), "mxfp8_quant_3d")
    return o


def device_status(reset: bool = False, stream=None):
    """(flags, fallbacks) of the current device; synchronizes the stream."""
    st, flags, n = capi.mxfp8_device_status(reset, _stream(stream))
    check(st, "mxfp8_device_status")
    return flags, n
