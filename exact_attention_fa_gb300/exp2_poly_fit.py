"""Coefficients of the software exponential (exp2_poly2 in csrc/fa_ptx.cuh).

2^f on [-1/2, 1/2] by a degree-3 polynomial that minimises the maximum relative error, found with
the Remez exchange algorithm: solve for the coefficients and the levelled error on n = degree + 2
reference points, move the points to the extrema of the error, repeat. The kernel splits x into
j + f (j = rint(x)) and scales the polynomial by 2^j, so this interval covers every input.

    python -m exact_attention_fa_gb300.exp2_poly_fit     # prints the coefficients and the error
"""
from __future__ import annotations

import numpy as np


def remez_exp2(degree: int = 3, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    """(coefficients c_0 .. c_degree, max relative error) of the minimax fit of 2^f."""
    n = degree + 2
    k = np.arange(n)
    x = (lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * k[::-1] / (n - 1))  # Chebyshev start
    grid = np.linspace(lo, hi, 200001)
    c = None
    err = np.inf
    for _ in range(iters):
        a = np.zeros((n, n))
        a[:, :degree + 1] = x[:, None] ** np.arange(degree + 1)
        a[:, degree + 1] = (-1.0) ** k * 2.0 ** x  # levelled relative error, alternating sign
        sol = np.linalg.solve(a, 2.0 ** x)
        c = sol[:degree + 1]
        e = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        err = float(np.abs(e).max())
        segments = np.split(np.arange(grid.size), np.where(np.diff(np.sign(e)) != 0)[0] + 1)
        extrema = np.array([grid[seg[np.argmax(np.abs(e[seg]))]] for seg in segments])
        if extrema.size != n:
            break
        x = extrema
    return c, err


def fp32_horner_error(c32: np.ndarray, lo: float = -0.5, hi: float = 0.5, points: int = 1000001):
    """Max relative error of the fp32 coefficients evaluated by fp32 Horner with fused
    multiply-adds (each step computed exactly, then rounded to fp32, as the kernel's fma does)."""
    f = np.linspace(lo, hi, points).astype(np.float32)
    r = np.float32(c32[-1]) * np.ones_like(f)
    for cc in c32[-2::-1]:
        r = (r.astype(np.float64) * f.astype(np.float64) + np.float64(cc)).astype(np.float32)
    exact = 2.0 ** f.astype(np.float64)
    return float(np.abs((r.astype(np.float64) - exact) / exact).max())


if __name__ == "__main__":
    coef, e = remez_exp2()
    c32 = coef.astype(np.float32)
    print("coefficients:", [float(v) for v in c32])
    print(f"minimax relative error {e:.3e}; fp32 Horner {fp32_horner_error(c32):.3e}")
