"""Layout invariants of the oracle's 2D and 3D quantizers.

* "both" equals rowwise-only plus colwise-only (the cross-mode consistency
  check of "Add swiglu + MXFP8 fused CuTe DSL kernel", section "Numerics and
  tests");
* colwise(X) is rowwise(X^T) transposed (a transposed operand or a wrong
  leading dimension in either loop nest fails this);
* the 3D per-expert colwise quantizer equals the 2D colwise quantizer on
  each expert's slab ("[mxfp8 moe training] update 3d quant colwise scaling
  kernel ...", section "Summary": column major per expert);
* row-range restriction computes exactly the selected rows.
"""
import numpy as np
import torch

import oracle as O


def rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * std).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def test_both_equals_row_plus_col():
    x = rand_bf16((96, 160), 1)
    b = O.quant_2d(x, O.BOTH)
    r = O.quant_2d(x, O.ROWWISE)
    c = O.quant_2d(x, O.COLWISE)
    for k in ("q_row", "s_row"):
        assert np.array_equal(b[k], r[k])
    for k in ("q_col", "s_col"):
        assert np.array_equal(b[k], c[k])


def test_colwise_is_rowwise_of_transpose():
    x = rand_bf16((128, 96), 2)
    c = O.quant_2d(x, O.COLWISE)
    r = O.quant_2d(np.ascontiguousarray(x.T), O.ROWWISE)
    assert np.array_equal(c["q_col"], r["q_row"])          # (N, M) both
    assert np.array_equal(c["s_col"], r["s_row"].T)


def test_quant_3d_equals_per_expert_2d_colwise():
    E, N, K = 3, 64, 48
    x = rand_bf16((E, N, K), 3, std=0.02)
    q, s = O.quant_3d_colwise(x)
    for e in range(E):
        c = O.quant_2d(np.ascontiguousarray(x[e]), O.COLWISE)
        assert np.array_equal(q[e], c["q_col"])             # (K, N)
        assert np.array_equal(s[e], c["s_col"])             # (N/32, K)


def test_row_range_restriction():
    x = rand_bf16((128, 64), 4)
    full = O.quant_2d(x, O.BOTH)
    part = O.quant_2d(x, O.BOTH, rows=(32, 96))
    assert np.array_equal(part["q_row"][32:96], full["q_row"][32:96])
    assert not part["q_row"][:32].any()
    assert np.array_equal(part["q_col"][:, 32:96], full["q_col"][:, 32:96])
    assert np.array_equal(part["s_col"][1:3], full["s_col"][1:3])


def test_strided_input_ld_larger_than_n():
    big = rand_bf16((64, 128), 5)
    view = big[:, 32:96]                                     # ld = 128, N = 64
    a = O.quant_2d(view, O.BOTH)
    b = O.quant_2d(np.ascontiguousarray(view), O.BOTH)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_bwd_grads_shapes_and_threads_do_not_change_results():
    dh, g, u = rand_bf16((64, 64), 6), rand_bf16((64, 64), 7), rand_bf16((64, 64), 8)
    a = O.swiglu_bwd_grads(dh, g, u, threads=1)
    b = O.swiglu_bwd_grads(dh, g, u, threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
