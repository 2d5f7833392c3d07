"""Derive the polynomial the prefill softmax uses for part of its base-2 exponentials.

2^f on [-1/2, 1/2] is approximated by p(f) = c0 + c1 f + ... + cn f^n, minimising the maximum
RELATIVE error with the Remez exchange algorithm (equioscillation of the weighted error
(p(f) - 2^f) / 2^f at n + 2 points).  The kernel evaluates p with Horner's rule in fp32 after
splitting a = j + f (j = nearest integer) and then adds j to the exponent field, so
2^a = 2^j * p(f).

Run: python derive_exp2_poly.py [degree]   (prints the coefficients and the error bound)
"""
import sys

import numpy as np


def remez_exp2(degree: int, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    n = degree
    # start from Chebyshev extrema
    k = np.arange(n + 2)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k / (n + 1))[::-1]
    grid = np.linspace(lo, hi, 200001)
    coef = None
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i  for c_0..c_n, E
        A = np.zeros((n + 2, n + 2))
        for i, xi in enumerate(x):
            A[i, : n + 1] = xi ** np.arange(n + 1)
            A[i, n + 1] = -((-1) ** i) * 2.0 ** xi
        sol = np.linalg.solve(A, 2.0 ** x)
        coef = sol[: n + 1]
        err = (np.polyval(coef[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: extrema of the error between sign changes
        sign = np.sign(err)
        idx = [0]
        for i in range(1, len(grid)):
            if sign[i] != sign[idx[-1]] and sign[i] != 0:
                idx.append(i)
            elif abs(err[i]) > abs(err[idx[-1]]):
                idx[-1] = i
        if len(idx) < n + 2:
            break
        # keep the n + 2 largest alternating extrema
        idx = np.array(idx)
        while len(idx) > n + 2:
            if abs(err[idx[0]]) < abs(err[idx[-1]]):
                idx = idx[1:]
            else:
                idx = idx[:-1]
        x = grid[idx]
    err = (np.polyval(coef[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
    return coef, float(np.abs(err).max())


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c, e = remez_exp2(deg)
    c32 = c.astype(np.float32)
    g = np.linspace(-0.5, 0.5, 100001).astype(np.float32)
    p = np.zeros_like(g)
    for ci in c32[::-1]:
        p = p * g + ci
    e32 = float(np.abs((p.astype(np.float64) - 2.0 ** g.astype(np.float64)) / 2.0 ** g).max())
    print(f"degree {deg}: max relative error {e:.3e} (fp64 coefficients), {e32:.3e} (fp32 Horner)")
    for i, ci in enumerate(c32):
        print(f"  c{i} = {float(ci):.9e}f  ({float(ci).hex()})")
