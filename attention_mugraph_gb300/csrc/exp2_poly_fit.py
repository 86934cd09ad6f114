"""Fit the polynomial used for 2^f on f in [-1/2, 1/2] by the FMA-pipe exponential.

Method: 2^x = 2^r * 2^f with r = round-to-nearest(x) and f = x - r in [-1/2, 1/2] (the
classic additive range reduction, exact in fp32 for |x| < 2^22), then a polynomial for 2^f
whose coefficients minimise the maximum RELATIVE error on [-1/2, 1/2] (Remez exchange,
implemented below from the equioscillation theorem). The kernel evaluates the polynomial by
Horner's rule with fp32 fused multiply-adds and adds r to the exponent field.

Running this file prints the coefficients (as C hex floats, rounded to fp32) and the error of
the fp32 evaluation measured on a dense grid, emulating each fused multiply-add by an exact
double product-sum rounded once to fp32.
"""

from __future__ import annotations

import numpy as np

DEGREE = 5


def remez_relative(f, degree: int, lo: float, hi: float, iters: int = 30):
    """Minimax polynomial for f on [lo, hi] in relative error: minimise max |p/f - 1|."""
    n = degree + 2
    # Chebyshev extrema as the initial reference set.
    k = np.arange(n)
    x = (lo + hi) / 2 + (hi - lo) / 2 * -np.cos(np.pi * k / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    coef = None
    for _ in range(iters):
        # Solve p(x_i) - (-1)^i E f(x_i) = f(x_i) for the coefficients and the level E.
        A = np.zeros((n, n))
        for j in range(degree + 1):
            A[:, j] = x ** j
        A[:, degree + 1] = -((-1.0) ** k) * f(x)
        sol = np.linalg.solve(A, f(x))
        coef = sol[: degree + 1]
        err = np.polyval(coef[::-1], grid) / f(grid) - 1.0
        # New reference: the extremum of each sign-constant run of the error.
        sign = np.sign(err)
        breaks = np.nonzero(np.diff(sign) != 0)[0] + 1
        runs = np.split(np.arange(grid.size), breaks)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) < n:
            break
        # Keep n alternating extrema with the largest magnitudes (contiguous window).
        best, best_val = None, -1.0
        for s in range(len(ext) - n + 1):
            win = ext[s:s + n]
            v = np.min(np.abs(err[win]))
            if v > best_val:
                best, best_val = win, v
        x = grid[best]
    return coef


def fp32(v):
    return np.float32(v)


def horner_fp32(coef32, f32):
    """Horner's rule with each step a fused multiply-add rounded once to fp32."""
    p = np.full_like(f32, coef32[-1], dtype=np.float32)
    for c in coef32[-2::-1]:
        p = (p.astype(np.float64) * f32.astype(np.float64) + np.float64(c)).astype(np.float32)
    return p


def exp2_emulated(x32, coef32):
    """The kernel's steps in fp32: round-to-nearest via the 1.5*2^23 shifter, f = x - r,
    polynomial, then r added to the exponent field."""
    x32 = np.maximum(x32, np.float32(-125.0))
    shifter = np.float32(12582912.0)
    t = (x32 + shifter).astype(np.float32)
    r = (t - shifter).astype(np.float32)
    f = (x32 - r).astype(np.float32)
    p = horner_fp32(coef32, f)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.astype(np.int32).view(np.float32)


def fit(degree: int = DEGREE):
    coef = remez_relative(np.exp2, degree, -0.5, 0.5)
    return np.array([fp32(c) for c in coef], dtype=np.float32)


def max_rel_error(coef32, lo=-30.0, hi=12.0, n=2_000_001):
    x = np.linspace(lo, hi, n).astype(np.float32)
    y = exp2_emulated(x, coef32).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    return float(np.max(np.abs(y / ref - 1.0)))


if __name__ == "__main__":
    c = fit()
    for i, v in enumerate(c):
        print(f"c{i} = {float(v).hex()}f  /* {float(v):.9g} */")
    print(f"max relative error of the fp32 evaluation on [-30, 12]: {max_rel_error(c):.3e}")
