#!/usr/bin/env python3
"""Fits the polynomial behind the attention kernel's FMA-pipe exp2 and prints its
coefficients (the constants in exp2_fma.cuh come from this script).

Method (Cody and Waite style range reduction, then a minimax polynomial):
    2^x = 2^n * 2^f,  n = round(x),  f = x - n in [-1/2, 1/2],
    2^f ~ p(f) = c0 + c1 f + ... + cd f^d,
with p chosen by the Remez exchange algorithm to minimise the maximum RELATIVE error
|p(f) / 2^f - 1| on [-1/2, 1/2] (weighted minimax: error function e(f) = p(f) 2^-f - 1).
The coefficients are then rounded to fp32 and the error re-measured in fp64.

Run: python gen_exp2_poly.py [degree]
"""
from __future__ import annotations

import sys

import numpy as np


def remez_exp2(degree: int, iters: int = 60):
    lo, hi = -0.5, 0.5
    n = degree + 2                                   # reference points
    k = np.arange(n)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n - 1 - k) / (n - 1))   # Chebyshev extrema
    grid = np.linspace(lo, hi, 200001)
    c = None
    for _ in range(iters):
        # Solve p(x_i) 2^-x_i - 1 = (-1)^i E  for c_0..c_d and E.
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :degree + 1] = (x[i] ** np.arange(degree + 1)) * 2.0 ** (-x[i])
            A[i, degree + 1] = -((-1.0) ** i)
        sol = np.linalg.solve(A, np.ones(n))
        c = sol[:degree + 1]
        err = np.polyval(c[::-1], grid) * 2.0 ** (-grid) - 1.0
        # New reference: the extrema of err between its sign changes.
        sign = np.sign(err)
        idx = np.where(np.diff(sign) != 0)[0]
        bounds = np.concatenate([[0], idx + 1, [len(grid)]])
        ext = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            seg = np.abs(err[a:b])
            ext.append(a + int(np.argmax(seg)))
        if len(ext) != n:
            # keep the n largest alternating extrema
            ext = sorted(sorted(ext, key=lambda i: -abs(err[i]))[:n])
            if len(ext) != n:
                break
        x_new = grid[ext]
        if np.max(np.abs(x_new - x)) < 1e-12:
            x = x_new
            break
        x = x_new
    return c


def max_rel_error(c, fp32=True):
    cc = np.asarray(c, dtype=np.float32 if fp32 else np.float64).astype(np.float64)
    f = np.linspace(-0.5, 0.5, 2000001)
    return float(np.max(np.abs(np.polyval(cc[::-1], f) * 2.0 ** (-f) - 1.0)))


def main():
    degree = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c = remez_exp2(degree)
    c32 = np.asarray(c, dtype=np.float32)
    print(f"degree {degree}: max relative error {max_rel_error(c, False):.3e} (fp64 coefficients), "
          f"{max_rel_error(c32):.3e} (fp32 coefficients)")
    for i, v in enumerate(c32):
        print(f"  c{i} = {float(v)!r:>24}  ({float(v).hex()})")


if __name__ == "__main__":
    main()
