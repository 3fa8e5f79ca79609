"""Minimax polynomial for 2^f on [-1/2, 1/2], used by the attention kernels
to compute part of the softmax exponentials on the FMA pipe.

Method: range reduction x = n + f with n = round-to-nearest(x) (adding and
subtracting 1.5 * 2^23 in fp32 rounds to an integer), so f lies in
[-1/2, 1/2]; 2^x = 2^n * p(f), the factor 2^n applied by adding n to the
exponent field.  p is the degree-3 polynomial minimising the maximum
relative error |p(f) / 2^f - 1| on [-1/2, 1/2], found by the Remez exchange
algorithm (alternation of the error at n + 2 points), written here from the
algorithm's definition.  The coefficients are rounded to fp32, and the error
is measured again with fp32 arithmetic (fused multiply-adds in Horner form).

Running this file prints the coefficients the kernels hold
(`csrc/varlen_fwd_kernel.cuh`, kExp2C0 .. kExp2C3) and the measured error bound; the
CPU test `tests/test_exp2_poly.py` checks those constants against this fit
and the error against the bound.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def remez(degree: int = DEGREE, lo: float = LO, hi: float = HI, iters: int = 50):
    """Coefficients c[0..degree] (c[k] multiplies f^k) of the relative-error
    minimax fit of 2^f on [lo, hi], and the levelled error E."""
    n = degree
    k = np.arange(n + 2)
    # Start from Chebyshev extrema mapped to the interval.
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n + 1 - k) / (n + 1))
    grid = np.linspace(lo, hi, 200001)
    E = 0.0
    c = np.zeros(n + 1)
    for _ in range(iters):
        # Solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for c and E.
        A = np.zeros((n + 2, n + 2))
        for i, xi in enumerate(x):
            A[i, : n + 1] = xi ** np.arange(n + 1)
            A[i, n + 1] = -((-1) ** i) * 2.0 ** xi
        sol = np.linalg.solve(A, 2.0 ** x)
        c, E = sol[: n + 1], sol[n + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # New reference: the extremum of the error in each sign-alternating
        # segment, keeping the end points.
        sign = np.sign(err)
        idx = [0]
        for j in range(1, grid.size):
            if sign[j] != sign[idx[-1]] and sign[j] != 0:
                idx.append(j)
            elif abs(err[j]) > abs(err[idx[-1]]):
                idx[-1] = j
        if len(idx) < n + 2:
            break
        # Keep n + 2 alternating extrema with the largest error.
        while len(idx) > n + 2:
            drop = 0 if abs(err[idx[0]]) < abs(err[idx[-1]]) else len(idx) - 1
            idx.pop(drop)
        new_x = grid[idx]
        if np.allclose(new_x, x, atol=1e-12):
            break
        x = new_x
    return c, abs(E)


def fp32_coefficients(c):
    return np.asarray(c, dtype=np.float32)


def eval_fp32(c32, x):
    """2^x for fp32 x the way the kernels compute it: x clamped at -125 (so
    that the exponent stays normal), fp32 rounding to the nearest integer
    with 1.5 * 2^23, Horner form with fused multiply-adds (each exact in
    double, then rounded once to fp32), and the exponent added to the bit
    pattern."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c32[-1])
    for ck in c32[-2::-1]:
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(ck)).astype(np.float32)
    bits = p.view(np.uint32).astype(np.int64) + (n.astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def max_rel_error(c32, lo=-125.0, hi=8.0, samples=2_000_001):
    x = np.linspace(lo, hi, samples, dtype=np.float64).astype(np.float32)
    got = eval_fp32(c32, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    return float(np.max(np.abs(got / ref - 1.0)))


if __name__ == "__main__":
    c, E = remez()
    c32 = fp32_coefficients(c)
    print("levelled relative error (exact coefficients):", E)
    print("fp32 coefficients c0..c3:", [float(v) for v in c32])
    print("as C literals:", ", ".join(f"{float(v):.9e}f" for v in c32))
    print("max relative error in fp32 on [-125, 8]:", max_rel_error(c32))
