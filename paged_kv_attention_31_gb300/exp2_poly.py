"""Coefficients of the polynomial the prefill kernel uses for part of its
2^x evaluations (on the FMA pipe, beside the hardware's ex2).

2^x is split as 2^r * 2^f with r = round(x) and f = x - r in [-1/2, 1/2];
2^r goes into the exponent bits, and 2^f is a polynomial p(f).  The
coefficients below minimise the largest relative error |p(f) / 2^f - 1| over
[-1/2, 1/2] (Remez exchange on the equioscillating error; degree 3 gives
about 7.5e-5, far below the 2^-9 relative rounding of the bf16 (2^-12 for
f16) P values the kernel stores).  Run as a script to print them.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _solve(nodes: np.ndarray, deg: int):
    """Polynomial c (lowest first) and level E with p(x_i) - 2^x_i =
    (-1)^i E 2^x_i at the deg + 2 nodes."""
    n = deg + 2
    a = np.zeros((n, n))
    for i, x in enumerate(nodes):
        a[i, :deg + 1] = x ** np.arange(deg + 1)
        a[i, deg + 1] = -((-1) ** i) * 2.0 ** x
    sol = np.linalg.solve(a, 2.0 ** nodes)
    return sol[:deg + 1], sol[deg + 1]


def _rel_err(c: np.ndarray, xs: np.ndarray) -> np.ndarray:
    return np.polyval(c[::-1], xs) / 2.0 ** xs - 1.0


def minimax(deg: int = DEGREE, iters: int = 40, grid: int = 400001):
    """Remez exchange for the relative error of p ~ 2^x on [LO, HI].
    Returns (coefficients lowest first, max relative error on the grid)."""
    n = deg + 2
    nodes = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * (np.arange(n)[::-1] + 0.5) / n)
    xs = np.linspace(LO, HI, grid)
    c = None
    for _ in range(iters):
        c, _ = _solve(nodes, deg)
        err = _rel_err(c, xs)
        # the n alternating extrema of the error: split the grid at sign
        # changes and keep the largest |err| of each run (ends included)
        sign = np.sign(err)
        cuts = np.flatnonzero(sign[1:] != sign[:-1]) + 1
        runs = np.split(np.arange(grid), cuts)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        while len(ext) > n:  # drop the smaller end extremum
            ext.pop(0 if abs(err[ext[0]]) < abs(err[ext[-1]]) else -1)
        if len(ext) < n:
            break
        nodes = xs[ext]
    return c, float(np.max(np.abs(_rel_err(c, xs))))


def coefficients_f32():
    """The coefficients rounded to float32 (c0 first), as the kernel holds them."""
    c, _ = minimax()
    return [float(np.float32(v)) for v in c]


if __name__ == "__main__":
    c, e = minimax()
    print(f"degree {DEGREE}, max relative error {e:.3e}")
    for i, v in enumerate(c):
        print(f"c{i} = {float(np.float32(v)).hex()}  ({np.float32(v)!r})")
