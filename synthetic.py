"""Seeded synthetic bf16 inputs for the MXFP8 cast workloads.

This module draws random tensors and nothing else: it holds none of the
cast's arithmetic, so the CUDA path and the CPU oracle can both be fed from
it.  Every tensor is drawn in fp32 by a seeded ``torch.Generator`` on the
requested device, scaled, and rounded to bf16 (round to nearest even).  The
same seed on the same device type gives the same bytes; tests that compare
the GPU path with the oracle draw once and copy the bytes to the host.

Workloads (shapes and value mixes of the pages' benchmark tables:
"Add swiglu + MXFP8 fused CuTe DSL kernel", section "Performance", and
"[mxfp8 moe training] update 3d quant colwise scaling kernel ...", section
"Performance"):

* ``fwd_128x128`` (seed 0): one (128, 256) buffer of N(0, 1); gate is
  columns 0..127, up is columns 128..255 (the packed ``[gate | up]`` layout
  of a fused w13 projection).
* ``mixed_4096x7168`` (seed 1): gate, up, dh each (4096, 7168) N(0, 1);
  in every tensor the rows i with i % 7 == 0 are multiplied by 2^k, k drawn
  uniformly from the integers -20..20 per row; then 1% of the 1x32 row
  blocks and 1% of the 32x1 column blocks are set to zero.
* ``outlier_16384x7168`` (seed 2): gate ~ N(0, 2^2), up ~ N(0, 1),
  dh ~ N(0, 0.01^2) (the second parameter read as the standard deviation);
  in 0.1% of the 1x32 row blocks of each tensor one element, at a uniformly
  drawn position, is set to +-1e4 (bf16 9984).
* ``large_131072x8192`` (seed 3): gate, up, dh each (131072, 8192) N(0, 1).
* ``experts_E`` (seed 4): (E, 8192, 5120) N(0, 0.02^2) expert weights.
"""
from __future__ import annotations

import torch

SEEDS = {
    "fwd_128x128": 0,
    "mixed_4096x7168": 1,
    "outlier_16384x7168": 2,
    "large_131072x8192": 3,
    "experts": 4,
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def fwd_128x128(device="cpu"):
    """Returns (buf (128, 256), gate view, up view)."""
    gen = _gen(SEEDS["fwd_128x128"], device)
    buf = normal_bf16((128, 256), 1.0, gen, device)
    return buf, buf[:, :128], buf[:, 128:]


def _scale_rows_pow2(x: torch.Tensor, gen: torch.Generator, every: int = 7, kmax: int = 20):
    M = x.shape[0]
    rows = torch.arange(0, M, every, device=x.device)
    k = torch.randint(-kmax, kmax + 1, (rows.numel(),), generator=gen, device=x.device)
    f = torch.pow(2.0, k.to(torch.float32)).to(torch.bfloat16)   # exact powers of two
    x[rows] = (x[rows].float() * f.float()[:, None]).to(torch.bfloat16)


def _zero_blocks(x: torch.Tensor, gen: torch.Generator, frac: float):
    M, N = x.shape
    # 1x32 row blocks
    if N % 32 == 0:
        m = torch.rand((M, N // 32), generator=gen, device=x.device) < frac
        x.view(M, N // 32, 32).masked_fill_(m[:, :, None], 0)
    # 32x1 column blocks
    if M % 32 == 0:
        m = torch.rand((M // 32, N), generator=gen, device=x.device) < frac
        x.view(M // 32, 32, N).masked_fill_(m[:, None, :], 0)


def mixed(M=4096, N=7168, device="cpu", seed=None):
    """gate, up, dh with power-of-two row scaling and zeroed 32-blocks."""
    gen = _gen(SEEDS["mixed_4096x7168"] if seed is None else seed, device)
    out = []
    for _ in range(3):
        x = normal_bf16((M, N), 1.0, gen, device)
        _scale_rows_pow2(x, gen)
        _zero_blocks(x, gen, 0.01)
        out.append(x)
    return tuple(out)   # gate, up, dh


def _plant_outliers(x: torch.Tensor, gen: torch.Generator, frac: float, mag: float = 1e4):
    M, N = x.shape
    m = torch.rand((M, N // 32), generator=gen, device=x.device) < frac
    pos = torch.randint(0, 32, (M, N // 32), generator=gen, device=x.device)
    sgn = torch.randint(0, 2, (M, N // 32), generator=gen, device=x.device) * 2 - 1
    r, b = torch.nonzero(m, as_tuple=True)
    c = b * 32 + pos[r, b]
    x[r, c] = (sgn[r, b].to(torch.float32) * mag).to(torch.bfloat16)


def outlier(M=16384, N=7168, device="cpu", seed=None):
    """gate ~ N(0,4), up ~ N(0,1), dh ~ N(0,1e-4), +-1e4 in 0.1% of row blocks."""
    gen = _gen(SEEDS["outlier_16384x7168"] if seed is None else seed, device)
    gate = normal_bf16((M, N), 2.0, gen, device)
    up = normal_bf16((M, N), 1.0, gen, device)
    dh = normal_bf16((M, N), 1e-2, gen, device)
    for x in (gate, up, dh):
        _plant_outliers(x, gen, 1e-3)
    return gate, up, dh


def large(M=131072, N=8192, device="cpu", seed=None):
    """gate, up, dh each N(0, 1)."""
    gen = _gen(SEEDS["large_131072x8192"] if seed is None else seed, device)
    return tuple(normal_bf16((M, N), 1.0, gen, device) for _ in range(3))


def experts(E, N=8192, K=5120, device="cpu", seed=None):
    """(E, N, K) expert weights ~ N(0, 0.02^2), row-major."""
    gen = _gen(SEEDS["experts"] if seed is None else seed, device)
    return normal_bf16((E, N, K), 0.02, gen, device)


def packed_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """[gate | up] as one (M, 2N) buffer (the fused w13 output layout)."""
    return torch.cat([gate, up], dim=1)
