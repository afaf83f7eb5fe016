"""The oracle's per-group blocked scale layouts, checked on the CPU against
the plain blocked layout (itself pinned on the GPU by driving a block-scaled
GEMM, tests/test_gpu_blocked.py) through what a grouped GEMM reads:

* M-groups (row scales of token groups): group g's 128-row tiles, taken
  alone, are exactly the plain blocked layout of the group's own rows -- the
  scale operand a per-group GEMM of that group's rows reads -- and they
  start right after the previous group's tiles; everything else is zero.
* K-groups (column scales, the (N, M/32) matrix, tokens along the columns):
  group g's 4-column tiles, cut out of every tile row and put together, are
  the plain blocked layout of the group's own columns; everything else zero.
* per-expert 3D: every expert's region is the plain layout of its matrix,
  and for uniform groups the M-groups layout agrees with it (two separately
  written functions).
Group-end vectors include empty groups and ragged sizes.
"""
import numpy as np
import pytest

import oracle as O


def _ceil(a, b):
    return -(-a // b)


def _labels(R, C, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(1, 256, (R, C)).astype(np.uint8)


def _tiles(flat, tiles_c):
    """flat blocked bytes -> (tile rows, tiles_c, 512)"""
    return flat.reshape(-1, tiles_c, 512)


@pytest.mark.parametrize("ends", [[300], [100, 300], [0, 128, 128, 260, 300], [32, 64, 96, 300]])
def test_m_groups_each_group_is_its_own_blocked_matrix(ends):
    R, C = 300, 7
    s = _labels(R, C, len(ends))
    got = O.scales_blocked_m_groups(s, ends)
    tiles_c = _ceil(C, 4)
    assert got.size == (_ceil(R, 128) + len(ends)) * 128 * tiles_c * 4
    t = _tiles(got, tiles_c)
    used = np.zeros(t.shape[0], bool)
    row_tile, start = 0, 0
    for end in ends:
        n = end - start
        k = _ceil(n, 128)
        if n:
            want = O.scales_blocked(s[start:end])
            assert np.array_equal(t[row_tile:row_tile + k].reshape(-1), want)
        used[row_tile:row_tile + k] = True
        row_tile += k
        start = end
    assert not t[~used].any()
    # every label once (multiset of the non-padding bytes)
    assert np.array_equal(np.sort(got[got != 0]), np.sort(s.reshape(-1)))


@pytest.mark.parametrize("ends", [[256], [96, 256], [0, 32, 32, 160, 256], [128, 256]])
def test_k_groups_each_group_is_its_own_blocked_matrix(ends):
    N, M = 200, 256
    s = _labels(N, M // 32, 10 + len(ends))          # the (N, M/32) matrix
    got = O.scales_blocked_k_groups(s, ends)
    tiles_c = _ceil(M, 128) + len(ends)
    assert got.size == _ceil(N, 128) * tiles_c * 512
    t = _tiles(got, tiles_c)
    used = np.zeros(tiles_c, bool)
    col_tile, start = 0, 0
    for end in ends:
        ca, cb = start // 32, end // 32
        k = _ceil(cb - ca, 4)
        if cb > ca:
            want = O.scales_blocked(s[:, ca:cb])
            assert np.array_equal(t[:, col_tile:col_tile + k].reshape(-1), want)
        used[col_tile:col_tile + k] = True
        col_tile += k
        start = end
    assert not t[:, ~used].any()
    assert np.array_equal(np.sort(got[got != 0]), np.sort(s.reshape(-1)))


@pytest.mark.parametrize("E,N,C", [(3, 96, 5), (2, 128, 4), (4, 160, 9)])
def test_per_expert_layout_matches_uniform_m_groups(E, N, C):
    s = _labels(E * N, C, E * N + C)
    per = O.scales_blocked_per_expert(s.reshape(E, N, C))
    assert per.size == E * _ceil(N, 128) * 128 * _ceil(C, 4) * 4
    for e in range(E):
        sz = per.size // E
        assert np.array_equal(per[e * sz:(e + 1) * sz], O.scales_blocked(s[e * N:(e + 1) * N]))
    mg = O.scales_blocked_m_groups(s, [N * (e + 1) for e in range(E)])
    assert np.array_equal(mg[:per.size], per)
    assert not mg[per.size:].any()


def test_group_end_rules():
    s = np.ones((64, 2), np.uint8)
    with pytest.raises(AssertionError):
        O.scales_blocked_m_groups(s, [32, 60])           # last end must be R
    with pytest.raises(AssertionError):
        O.scales_blocked_m_groups(s, [40, 30, 64])       # not non-decreasing
    with pytest.raises(AssertionError):
        O.scales_blocked_k_groups(np.ones((8, 2), np.uint8), [40, 64])   # K-groups need 32-row ends


@pytest.mark.parametrize("M,N,ends", [(416, 160, [96, 96, 224, 416]), (1024, 288, [32, 160, 480, 992, 1024]),
                                      (640, 4256, [640]), (400, 96, [64, 64, 320, 400])])
def test_binding_allocates_the_oracle_layout_sizes(M, N, ends):
    """The Python binding sizes its zero-filled scale buffers from a formula;
    it must match the oracle's layouts byte for byte in length."""
    import mxfp8_quantization_moe_gb300 as mx
    rows = O.scales_blocked_m_groups(np.zeros((M, N // 32), np.uint8), ends).size
    rb, cb = mx.grouped_scale_bytes(M, N, len(ends))
    assert rb == rows
    if all(e % 32 == 0 for e in ends):
        cols = O.scales_blocked_k_groups(np.zeros((N, -(-M // 32)), np.uint8), ends).size
        assert cb == cols
    assert mx.blocked_bytes(M, N // 32) == O.scales_blocked(np.zeros((M, N // 32), np.uint8)).size
