"""GPU parity of the fused SwiGLU + MXFP8 forward and backward.

Tolerance (stated for the SwiGLU paths): E8M0 scales bit-exact; at most 1e-4
of the E4M3 codes may differ from the oracle, each by at most one code.  The
kernels keep a fast activation value (within one bf16 step of the correctly
rounded one) except where it could move a scale, so a few codes per million
may differ; every comparison checks the bound and the totals are printed.

Workloads: the packed (128, 128) forward; the (4096, 7168) mix of per-row
2^k scaling and zeroed 32-blocks (full comparison); the (16384, 7168)
outlier mix and the (131072, 8192) normal data compared on sampled 32-row
blocks; every bf16 gate value; amax at the E4M3 boundary.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import Guarded, bits, compare_codes, u8
import synthetic
from mxfp8_quantization_moe_gb300 import capi, device_status

pytestmark = pytest.mark.gpu

CODE_TOL = 1e-4


def _stream():
    return torch.cuda.current_stream().cuda_stream


def fwd_gpu(gate, up, mode, blocks=None, act="silu"):
    """Run the fused forward (act "gelu": GEGLU); return host outputs (only
    the 32-row blocks in `blocks` when given, gathered on the device)."""
    M, N = gate.shape
    o = {}
    if mode & 1:
        o["q_row"], o["s_row"] = Guarded((M, N)), Guarded((M, N // 32))
    if mode & 2:
        o["q_col"], o["s_col"] = Guarded((N, M)), Guarded((M // 32, N))
    p = lambda k: o[k].t.data_ptr() if k in o else None
    ld = lambda k: o[k].t.stride(0) if k in o else 0
    fn = capi.mxfp8_geglu_fwd if act == "gelu" else capi.mxfp8_swiglu_fwd
    st = fn(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
            p("q_row"), ld("q_row"), p("s_row"), ld("s_row"),
            p("q_col"), ld("q_col"), p("s_col"), ld("s_col"), _stream())
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    for k, g in o.items():
        assert g.intact(), k
    return gather({k: g.t for k, g in o.items()}, blocks)


def gather(d, blocks):
    """Device outputs -> host numpy, restricted to 32-row blocks if given."""
    if blocks is None:
        return {k: u8(t) for k, t in d.items()}
    sel = torch.tensor(rows_of(blocks), device="cuda")
    bl = torch.tensor(blocks, device="cuda")
    out = {}
    for k, t in d.items():
        if k in ("q_row", "s_row"):
            out[k] = u8(t.index_select(0, sel))
        elif k == "q_col":
            out[k] = u8(t.index_select(1, sel))
        else:
            out[k] = u8(t.index_select(0, bl))
    return out


def rows_of(blocks):
    return np.concatenate([np.arange(32 * b, 32 * b + 32) for b in blocks]).tolist()


def bwd_gpu(dh, gate, up, mode, blocks=None, act="silu"):
    """Packed [dGate | dUp] outputs; returns per-tensor dicts (dgate, dup)."""
    M, N = gate.shape
    o = {}
    if mode & 1:
        o["q_row"], o["s_row"] = Guarded((M, 2 * N)), Guarded((M, 2 * N // 32))
    if mode & 2:
        o["q_col"], o["s_col"] = Guarded((2 * N, M)), Guarded((M // 32, 2 * N))
    qr = o["q_row"].t.data_ptr() if mode & 1 else None
    sr = o["s_row"].t.data_ptr() if mode & 1 else None
    qc = o["q_col"].t.data_ptr() if mode & 2 else None
    sc = o["s_col"].t.data_ptr() if mode & 2 else None
    fn = capi.mxfp8_geglu_bwd if act == "gelu" else capi.mxfp8_swiglu_bwd
    st = fn(
        dh.data_ptr(), dh.stride(0), gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, mode,
        qr, qr + N if qr else None, 2 * N if qr else 0,
        sr, sr + N // 32 if sr else None, N // 16 if sr else 0,
        qc, qc + N * M if qc else None, M if qc else 0,
        sc, sc + N if sc else None, 2 * N if sc else 0, _stream())
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    for k, g in o.items():
        assert g.intact(), k
    t = {k: g.t for k, g in o.items()}
    dg, du = {}, {}
    if mode & 1:
        dg["q_row"], du["q_row"] = t["q_row"][:, :N], t["q_row"][:, N:]
        dg["s_row"], du["s_row"] = t["s_row"][:, :N // 32], t["s_row"][:, N // 32:]
    if mode & 2:
        dg["q_col"], du["q_col"] = t["q_col"][:N], t["q_col"][N:]
        dg["s_col"], du["s_col"] = t["s_col"][:, :N], t["s_col"][:, N:]
    return gather(dg, blocks), gather(du, blocks)


def compare(got, want, what=""):
    """Scales bit-exact; codes within tolerance.  Returns differing codes."""
    n = 0
    for k in want:
        g, w = np.ascontiguousarray(got[k]), np.ascontiguousarray(want[k])
        if k.startswith("s_"):
            assert np.array_equal(g, w), "%s %s: scales differ at %d places" % (what, k, int((g != w).sum()))
        else:
            d = compare_codes(g, w, CODE_TOL, what + " " + k)
            if d:
                print("%s %s: %d of %d codes differ by one" % (what, k, d, g.size))
            n += d
    return n


def _host_rows(t, blocks):
    if blocks is None:
        return bits(t)
    sel = torch.tensor(rows_of(blocks), device=t.device)
    return bits(t.index_select(0, sel))


ACTS = {"silu": O.SILU, "gelu": O.GELU}


def oracle_fwd(gate, up, mode, blocks=None, act="silu"):
    """Oracle on the whole tensors, or on the stacked 32-row blocks."""
    return O.swiglu_fwd(_host_rows(gate, blocks), _host_rows(up, blocks), mode, act=ACTS[act])[0]


def oracle_bwd(dh, gate, up, mode, blocks=None, act="silu"):
    r = O.swiglu_bwd(_host_rows(dh, blocks), _host_rows(gate, blocks), _host_rows(up, blocks), mode,
                     act=ACTS[act])
    return r[0], r[1]


# ------------------------------------------------------------ small shapes

def rand_inputs(M, N, seed, std=(2.0, 1.0, 0.05)):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return [(torch.randn((M, N), generator=g, device="cuda") * s).to(torch.bfloat16) for s in std]


@pytest.mark.parametrize("shape", [(32, 64), (160, 96), (256, 320), (1024, 576)], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_fwd_small(shape, mode):
    gate, up, _ = rand_inputs(*shape, seed=shape[0] + mode)
    got = fwd_gpu(gate, up, mode)
    compare(got, oracle_fwd(gate, up, mode), what="fwd")


@pytest.mark.parametrize("shape", [(32, 64), (160, 96), (256, 320), (1024, 576)], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_bwd_small(shape, mode):
    gate, up, dh = rand_inputs(*shape, seed=shape[1] + mode)
    dg, du = bwd_gpu(dh, gate, up, mode)
    wg, wu = oracle_bwd(dh, gate, up, mode)
    compare(dg, wg, what="dgate")
    compare(du, wu, what="dup")


def test_fwd_packed_128x128_rowwise():
    """The (128, 128) forward of the pages' sweep, [gate | up] in one buffer."""
    buf, gate, up = synthetic.fwd_128x128(device="cuda")
    for mode in (1, 2, 3):
        got = fwd_gpu(gate, up, mode)
        compare(got, oracle_fwd(gate, up, mode), what="fwd128")


# ----------------------------------------------------------- every gate

def every_gate(rows=512):
    v = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(rows, 65536 // rows)
    return torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("useed", [0, 1, 2])
def test_fwd_every_bf16_gate(useed):
    gate = every_gate()
    g = torch.Generator(device="cuda").manual_seed(100 + useed)
    up = (torch.randn(gate.shape, generator=g, device="cuda") *
          (1.0 if useed < 2 else 1e3)).to(torch.bfloat16)
    if useed == 1:
        up.fill_(1.0)
    for mode in (1, 2):
        got = fwd_gpu(gate, up, mode)
        compare(got, oracle_fwd(gate, up, mode), what="fwd-all-g")


@pytest.mark.parametrize("useed", [0, 1])
def test_bwd_every_bf16_gate(useed):
    gate = every_gate()
    g = torch.Generator(device="cuda").manual_seed(200 + useed)
    up = torch.randn(gate.shape, generator=g, device="cuda").to(torch.bfloat16)
    dh = (torch.randn(gate.shape, generator=g, device="cuda") * 0.01).to(torch.bfloat16)
    if useed == 1:
        up.fill_(1.0)
        dh.fill_(1.0)
    for mode in (1, 2):
        dg, du = bwd_gpu(dh, gate, up, mode)
        wg, wu = oracle_bwd(dh, gate, up, mode)
        compare(dg, wg, what="dgate-all-g")
        compare(du, wu, what="dup-all-g")


def test_fwd_amax_at_e4m3_boundary():
    """Blocks whose largest h sits next to 448 * 2^k: the scale byte flips
    there, so the bf16 rounding of h must match exactly."""
    M, N = 512, 256
    g = torch.Generator(device="cuda").manual_seed(7)
    gate = (torch.rand((M, N), generator=g, device="cuda") * 6 - 1).to(torch.bfloat16)
    up = (torch.randn((M, N), generator=g, device="cuda") * 0.1).to(torch.bfloat16)
    gf = gate.float()
    silu = gf * torch.sigmoid(gf)
    k = torch.randint(-10, 10, (M, N // 32), generator=g, device="cuda").float()
    target = 448.0 * torch.pow(2.0, k) * (1 + (torch.rand((M, N // 32), generator=g, device="cuda") - 0.5) * 0.02)
    pos = torch.randint(0, 32, (M, N // 32), generator=g, device="cuda")
    cols = torch.arange(N // 32, device="cuda") * 32 + pos
    rows = torch.arange(M, device="cuda")[:, None].expand_as(cols)
    s = silu[rows, cols]
    ok = s.abs() > 0.05
    u_new = torch.where(ok, target / s, up[rows, cols].float())
    up[rows, cols] = u_new.to(torch.bfloat16)
    for mode in (1, 2, 3):
        got = fwd_gpu(gate, up, mode)
        compare(got, oracle_fwd(gate, up, mode), what="fwd-boundary")


# ------------------------------------------------------- pages' workloads

def test_mixed_4096x7168_both_full():
    gate, up, dh = synthetic.mixed(device="cuda")
    got = fwd_gpu(gate, up, 3)
    n = compare(got, oracle_fwd(gate, up, 3), what="mixed fwd")
    dg, du = bwd_gpu(dh, gate, up, 3)
    wg, wu = oracle_bwd(dh, gate, up, 3)
    n += compare(dg, wg, what="mixed dgate") + compare(du, wu, what="mixed dup")
    print("differing codes:", n)


def sample_blocks(M, count, seed, edges=()):
    """`count` random 32-row blocks, the first and last, and `edges`."""
    rng = np.random.default_rng(seed)
    nb = M // 32
    pick = set(rng.choice(nb, size=min(count, nb), replace=False).tolist()) | {0, nb - 1}
    return sorted(pick | {b for b in edges if 0 <= b < nb})


def band_edges(M, tile_rows):
    """32-row blocks on both sides of tile-row boundaries: near the start,
    the middle and the end of the matrix, and the last (partial) band."""
    nb, per = M // 32, tile_rows // 32
    out = set()
    for t in (1, 2, (M // tile_rows) // 2, M // tile_rows - 1, M // tile_rows):
        out |= {t * per - 1, t * per}
    return sorted(b for b in out if 0 <= b < nb)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_outlier_16384x7168_sampled(mode):
    gate, up, dh = synthetic.outlier(device="cuda")
    rows = sample_blocks(gate.shape[0], 24, mode)
    got = fwd_gpu(gate, up, mode, rows)
    n = compare(got, oracle_fwd(gate, up, mode, rows), what="outlier fwd")
    dg, du = bwd_gpu(dh, gate, up, mode, rows)
    wg, wu = oracle_bwd(dh, gate, up, mode, rows)
    n += compare(dg, wg, what="outlier dgate") + compare(du, wu, what="outlier dup")
    print("differing codes:", n)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_large_131072x8192_sampled(mode):
    gate, up, dh = synthetic.large(device="cuda")
    M = gate.shape[0]
    # the forward's and the backward's tile heights (96, 128 rows)
    rows = sample_blocks(M, 40, 10 + mode, band_edges(M, 96) + band_edges(M, 128))
    got = fwd_gpu(gate, up, mode, rows)
    n = compare(got, oracle_fwd(gate, up, mode, rows), what="large fwd")
    dg, du = bwd_gpu(dh, gate, up, mode, rows)
    wg, wu = oracle_bwd(dh, gate, up, mode, rows)
    n += compare(dg, wg, what="large dgate") + compare(du, wu, what="large dup")
    print("differing codes:", n)


def _max_code_invariant(q, s, what):
    """RCEIL puts every block's largest magnitude in (224, 448] after the
    descale, so its largest code is 0x76..0x7E (for scale bytes 1..254);
    q (blocks, 32) codes, s (blocks,) scale bytes, on the device."""
    mag = (q & 0x7F).amax(dim=1)
    normal = (s > 0) & (s < 255)
    bad = normal & ((mag < 0x76) | (mag > 0x7E))
    assert int(bad.sum()) == 0, "%s: %d blocks break the largest-code rule" % (what, int(bad.sum()))
    nan_blocks = s == 255
    assert bool(((q[nan_blocks] & 0x7F) == 0x7F).all()), what


@pytest.mark.parametrize("kind", ["fwd", "bwd"])
def test_large_131072x8192_every_block_invariant(kind):
    """Every block of the (131072, 8192) casts, both directions, in the
    launch the benchmark times: the largest-code rule of RCEIL scales."""
    import mxfp8_quantization_moe_gb300 as mx
    gate, up, dh = synthetic.large(device="cuda")
    M, N = gate.shape
    outs = []
    if kind == "fwd":
        o = mx.swiglu_fwd(gate, up, 3)
        outs.append(("h", o.q_row, o.s_row, o.q_col, o.s_col))
    else:
        o = mx.swiglu_bwd(dh, gate, up, 3)
        for name, c in (("dgate", o.dgate()), ("dup", o.dup())):
            outs.append((name, c.q_row, c.s_row, c.q_col, c.s_col))
    torch.cuda.synchronize()
    for name, qr, sr, qc, sc in outs:
        _max_code_invariant(qr.reshape(M * N // 32, 32), sr.reshape(-1), name + " rowwise")
        # column-major data: column c's 32-row block b is q_col[c, 32b:32b+32]
        _max_code_invariant(qc.reshape(N * M // 32, 32), sc.t().reshape(-1), name + " colwise")
    flags, _ = device_status()
    assert flags == 0


def test_status_clean_and_fallback_path_used():
    flags, fallbacks = device_status()
    assert flags == 0
    assert fallbacks > 0      # the every-gate tests exercise the double path


@pytest.mark.parametrize("mode", [1, 3])
def test_fwd_with_h_writes_the_encoded_activation(mode):
    """The forward that also writes the bf16 activation: the casts as usual,
    and h within one bf16 step of the oracle's correctly rounded activation
    everywhere, equal to it in all but 1e-3 of the elements (the fast
    activation's error bound, 33 units of 2^-24, over a bf16 step of 2^-8,
    twice: 66 * 2^-16 ~ 1e-3); the codes are exactly the cast of that h."""
    M, N = 1024, 576
    gate, up, _ = rand_inputs(M, N, 31)
    import mxfp8_quantization_moe_gb300 as mx
    got = mx.swiglu_fwd(gate, up, mode, keep_h=True)
    torch.cuda.synchronize()
    want, h_want = O.swiglu_fwd(bits(gate), bits(up), mode)
    compare({k: u8(getattr(got, k)) for k in want}, want, what="fwd-with-h")
    h = bits(got.h)
    hv = (h.astype(np.uint32) << 16).view(np.float32)
    wv = (h_want.astype(np.uint32) << 16).view(np.float32)
    diff = h != h_want
    steps = np.abs(h.astype(np.int32) - h_want.astype(np.int32))[diff]
    assert np.all((np.sign(hv[diff]) == np.sign(wv[diff])) & (steps == 1)), "more than one bf16 step"
    assert diff.sum() <= 1e-3 * h.size, diff.sum()
    print("h differs from the correctly rounded activation at", int(diff.sum()), "of", h.size)
    # the rowwise codes are the standalone cast of the h written
    q = O.quant_2d(h, O.ROWWISE)
    assert np.array_equal(u8(got.q_row), q["q_row"]) and np.array_equal(u8(got.s_row), q["s_row"])


def test_fwd_with_h_ragged_rows_and_strided_h():
    """h leaves through TMA tensor stores of whole tiles: ragged rows (M not a
    multiple of the tile height), a ragged last column tile and an h row
    pitch wider than N -- h equals the oracle's within the fast-path
    tolerance, and nothing outside the (M, N) window of h is written."""
    M, N, LD = 1000, 320, 384
    gate, up, _ = rand_inputs(M, N, 37)
    hbuf = torch.full((M * LD + 2 * 4096,), 0x5A5A, dtype=torch.int16, device="cuda")
    hview = hbuf[4096:4096 + M * LD].view(M, LD)
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, N // 32), dtype=torch.uint8, device="cuda")
    st = capi.mxfp8_swiglu_fwd_with_h(gate.data_ptr(), up.data_ptr(), gate.stride(0), M, N, 1,
                                      hview.data_ptr(), LD, q.data_ptr(), N, s.data_ptr(), N // 32,
                                      None, 0, None, 0, _stream())
    assert st == 0, capi.STATUS_NAMES[st]
    torch.cuda.synchronize()
    hb = hbuf.cpu().numpy().view(np.uint16)
    assert np.all(hb[:4096] == 0x5A5A) and np.all(hb[4096 + M * LD:] == 0x5A5A), "h written outside its buffer"
    h = hb[4096:4096 + M * LD].reshape(M, LD)
    assert np.all(h[:, N:] == 0x5A5A), "h written beyond column N"
    want, h_want = O.swiglu_fwd(bits(gate), bits(up), 1)
    diff = h[:, :N] != h_want
    assert diff.sum() <= 1e-3 * M * N, diff.sum()
    steps = np.abs(h[:, :N].astype(np.int32) - h_want.astype(np.int32))[diff]
    assert np.all(steps == 1)
    compare({"q_row": u8(q), "s_row": u8(s)}, want, what="fwd-with-h-ragged")
