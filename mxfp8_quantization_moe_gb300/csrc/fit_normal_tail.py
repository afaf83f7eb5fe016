"""Fit of the rational normal tail used by GEGLU's second fast path (the
backward of the gated-activation kernels but for "both" with per-group
scales, device.cuh): for t >= 0,

    Phi(-t) = exp(-t^2 / 2) * z * R(z),   z = 1 / (1 + p t),

with R a polynomial of degree 7 whose coefficients minimise the largest
relative error of z R(z) against Phi(-t) exp(t^2 / 2) (the Mills ratio over
sqrt(2 pi)) on t in [0, 8], on a dense grid: a least-squares start, then the
minimax correction as a linear program (scaled so that the solver's
tolerances sit far below the error), p chosen by a scan.  Prints the constants for device.cuh (rounded to fp32).

Run on a host with SciPy:  python fit_normal_tail.py
"""
import numpy as np
from scipy.optimize import linprog
from scipy.special import log_ndtr

DEGREE = 7
T_MAX = 8.0


def target(t):
    return np.exp(log_ndtr(-t) + 0.5 * t * t)


def fit(p, n=DEGREE):
    t = np.unique(np.concatenate([np.linspace(0.0, T_MAX, 6000), np.geomspace(1e-5, T_MAX, 600)]))
    z = 1.0 / (1.0 + p * t)
    f = target(t)
    A = np.stack([z ** (k + 1) / f for k in range(n + 1)], 1)
    c0 = np.linalg.lstsq(A, np.ones(len(t)), rcond=None)[0]
    r0 = A @ c0 - 1.0
    scale = 2.0 ** 24                    # solve for scale * (c - c0) and scale * error
    m = len(t)
    cost = np.zeros(n + 2)
    cost[-1] = 1.0
    A_ub = np.block([[A, -np.ones((m, 1))], [-A, -np.ones((m, 1))]])
    b_ub = np.concatenate([-scale * r0, scale * r0])
    r = linprog(cost, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (n + 1) + [(0, None)], method="highs")
    c = c0 + r.x[:-1] / scale
    return c, np.abs(A @ c - 1.0).max()


def main():
    best = None
    for p in np.round(np.arange(0.22, 0.42, 0.005), 4):
        c, e = fit(float(np.float32(p)))
        if best is None or e < best[1]:
            best = (float(np.float32(p)), e, c)
    p, e, c = best
    print("// p = %.9g, max relative error of z R(z) on [0, %g]: %.3g (%.2f units of 2^-24)"
          % (p, T_MAX, e, e / 2.0 ** -24))
    print("constexpr float kTailP = %.9gf;" % p)
    print("constexpr float kTailR[%d] = {%s};" % (len(c), ", ".join("%.9gf" % np.float32(v) for v in c)))


if __name__ == "__main__":
    main()
