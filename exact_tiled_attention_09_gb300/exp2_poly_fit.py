"""Coefficients of the cubic that the backward kernel uses for part of its
exponentials (2^f on f in [-1/2, 1/2], minimax in relative error).

The kernel computes 2^x as 2^n * 2^f with n = round(x) and f = x - n in
[-1/2, 1/2] (range reduction to the nearest integer); 2^n goes into the
exponent field with an integer add, and 2^f is this polynomial, evaluated in
fp32 with fused multiply-adds (Horner).  The coefficients come from the
Remez exchange algorithm on the relative error 1 - p(f) / 2^f, run here in
float64; the result is rounded to fp32, the precision the kernel holds them
in.  Run this file to print them; the kernel's copies must match (a test
checks that).
"""

from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def remez_relative(degree=DEGREE, lo=LO, hi=HI, iters=30):
    """Minimax polynomial for 2^f under relative error on [lo, hi]."""
    n = degree + 2  # reference points
    k = np.arange(n)
    x = (lo + hi) / 2 + (hi - lo) / 2 * -np.cos(np.pi * k / (n - 1))  # Chebyshev extrema
    grid = np.linspace(lo, hi, 20001)
    coeffs = None
    for _ in range(iters):
        # p(x_i) - 2^{x_i} = (-1)^i E 2^{x_i}  ->  linear system in c_0..c_d, E
        f = np.exp2(x)
        A = np.zeros((n, n))
        for j in range(degree + 1):
            A[:, j] = x ** j
        A[:, degree + 1] = -((-1.0) ** k) * f
        sol = np.linalg.solve(A, f)
        coeffs = sol[:degree + 1]
        err = np.polyval(coeffs[::-1], grid) / np.exp2(grid) - 1.0
        # new reference: the extrema of the error, one per sign run
        idx = []
        sign = np.sign(err)
        start = 0
        for i in range(1, grid.size + 1):
            if i == grid.size or sign[i] != sign[start]:
                seg = slice(start, i)
                idx.append(start + int(np.argmax(np.abs(err[seg]))))
                start = i
        if len(idx) < n:
            break
        # keep the n largest alternating extrema
        while len(idx) > n:
            a = np.abs(err[idx])
            drop = 0 if a[0] < a[-1] else len(idx) - 1
            idx.pop(drop)
        x = grid[idx]
    return coeffs


def fp32_coefficients():
    return [float(np.float32(c)) for c in remez_relative()]


def max_relative_error(coeffs, samples=200001):
    """Max |p(f)/2^f - 1| on [-1/2, 1/2] with the kernel's fp32 Horner."""
    f = np.linspace(LO, HI, samples).astype(np.float32)
    c = [np.float32(v) for v in coeffs]
    p = np.full_like(f, c[-1])
    for v in c[-2::-1]:
        p = (p * f + v).astype(np.float32)  # fp32 products; the kernel fuses them
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    cs = fp32_coefficients()
    for i, c in enumerate(cs):
        print(f"c{i} = {c!r}  ({np.float32(c).view(np.uint32):#010x})")
    print("max relative error (fp32 Horner):", max_relative_error(cs))
