"""Derivation of the degree-3 polynomial the forward kernel uses for 2^f, f in [0, 1).

Remez exchange for the polynomial p minimising max |p(f) - 2^f| / 2^f on [0, 1)
(relative-error minimax).  Run it to reproduce the coefficients hard-coded in
csrc/sm100_ptx.cuh (``ex2_fma``) and their error bound; tests check the
committed float32 coefficients against the bound printed here.

    python -m attention_tiled_fwd_gb300.exp2_poly_fit
"""
from __future__ import annotations

import numpy as np

# float32 coefficients c0..c3 as committed in ex2_fma (p = c0 + c1 f + c2 f^2 + c3 f^3)
COEFFS = (0.99992520, 0.69583356, 0.22606716, 0.07802452)
MAX_REL_ERR = 7.5e-5


def remez(deg: int = 3, iters: int = 30, grid: int = 200001):
    n = deg + 2
    x = 0.5 - 0.5 * np.cos(np.pi * np.arange(n) / (n - 1))  # Chebyshev-like start
    g = np.linspace(0.0, 1.0, grid)
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * 2.0 ** x[i]  # equioscillating relative error
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], g) - 2.0 ** g) / 2.0 ** g
        d = np.diff(err)
        cand = [0] + [i for i in range(1, len(g) - 1) if (d[i - 1] > 0) != (d[i] > 0)] + [len(g) - 1]
        x = np.sort(g[sorted(cand, key=lambda i: -abs(err[i]))[:n]])
    return c, float(np.abs(err).max())


def max_rel_error(coeffs, grid: int = 400001) -> float:
    f = np.linspace(0.0, 1.0, grid)
    c = np.asarray(coeffs, dtype=np.float32).astype(np.float64)
    return float(np.abs(np.polyval(c[::-1], f) / 2.0 ** f - 1.0).max())


if __name__ == "__main__":
    c, e = remez()
    print("coefficients:", [float(np.float32(v)) for v in c], "max rel err %.3e" % e)
    print("committed float32 coefficients: max rel err %.3e" % max_rel_error(COEFFS))
