"""Helpers shared by the GPU parity tests (torch <-> numpy bit views, code
distance, guarded output buffers)."""
import numpy as np
import torch

import oracle as O

POISON = 0xA5
MARGIN = 4096


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_bf16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 keeping its row stride (for strided views)."""
    return bits(t)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def code_ordinal(c: np.ndarray) -> np.ndarray:
    """E4M3 code -> signed position on the number line (+0 and -0 both 0)."""
    c = c.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def compare_codes(got: np.ndarray, want: np.ndarray, max_frac: float, what: str):
    """Codes may differ in at most max_frac of elements, each by one code."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    diff = got != want
    n = int(diff.sum())
    if n:
        d = np.abs(code_ordinal(got[diff]) - code_ordinal(want[diff]))
        assert d.max() <= 1, "%s: a code differs by %d" % (what, int(d.max()))
    assert n <= max_frac * got.size, "%s: %d of %d codes differ" % (what, n, got.size)
    return n


class Guarded:
    """A uint8 device buffer with a poisoned margin on both sides."""

    def __init__(self, shape, device="cuda"):
        self.shape = tuple(shape)
        n = int(np.prod(self.shape))
        self.buf = torch.full((n + 2 * MARGIN,), POISON, dtype=torch.uint8, device=device)
        self.t = self.buf[MARGIN:MARGIN + n].view(self.shape)

    def intact(self) -> bool:
        b = self.buf
        return bool((b[:MARGIN] == POISON).all()) and bool((b[-MARGIN:] == POISON).all())


def oracle_quant(x_bits: np.ndarray, mode: int, rows=None):
    return O.quant_2d(x_bits, mode, rows=rows)
