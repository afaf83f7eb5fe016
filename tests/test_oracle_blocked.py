"""The oracle's blocked scale layout: structural checks on the CPU.

The order inside a 128 x 4 tile is a reading (the pages name the blocked
tcgen05 layout and its 128-row / 4-column padding, not the byte order); it
is pinned on the GPU by driving a block-scaled GEMM with the oracle's
blocked scales (tests/test_gpu_blocked.py).  Here: the transform moves every
entry exactly once, pads with zeros, keeps 128 x 4 tiles as contiguous
512-byte units in row-major tile order, and treats a transposed view like
the materialised transpose.
"""
import numpy as np
import pytest

import oracle as O


@pytest.mark.parametrize("R,C", [(1, 1), (32, 4), (128, 4), (130, 5), (300, 17), (96, 8)])
def test_every_entry_once_and_zero_padding(R, C):
    rng = np.random.default_rng(R * 31 + C)
    # distinct 16-bit labels split over two passes of 8-bit values
    idx = np.arange(R * C).reshape(R, C)
    lo = O.scales_blocked((idx % 251 + 1).astype(np.uint8))
    hi = O.scales_blocked((idx // 251 + 1).astype(np.uint8))
    rp, cp = -(-R // 128) * 128, -(-C // 4) * 4
    assert lo.size == rp * cp
    live = lo != 0
    assert live.sum() == R * C                      # padding entries are 0
    labels = (hi[live].astype(np.int64) - 1) * 251 + (lo[live].astype(np.int64) - 1)
    assert np.array_equal(np.sort(labels), np.arange(R * C))   # each entry exactly once


def test_tiles_are_contiguous_512_byte_units_in_row_major_tile_order():
    R, C = 384, 12                                  # 3 x 3 tiles
    s = np.zeros((R, C), np.uint8)
    for tr in range(3):
        for tc in range(3):
            s[tr * 128:(tr + 1) * 128, tc * 4:(tc + 1) * 4] = 1 + tr * 3 + tc
    b = O.scales_blocked(s)
    for t in range(9):
        assert np.all(b[t * 512:(t + 1) * 512] == 1 + t)


def test_transposed_view_equals_transposed_copy():
    rng = np.random.default_rng(3)
    s = rng.integers(0, 255, (40, 200), dtype=np.uint8)
    assert np.array_equal(O.scales_blocked(s.T), O.scales_blocked(np.ascontiguousarray(s.T)))
