"""Fits the polynomial behind the kernels' software exp2 (``exp2_poly2`` in
sm103_ptx.cuh) and prints its float32 coefficients.

2^x = 2^n * 2^f with n = round(x) and f in [-1/2, 1/2] (the range reduction
of Cody and Waite, "Software Manual for the Elementary Functions", 1980,
which for base 2 needs no split constant). 2^f is approximated by the
degree-3 polynomial that minimises the maximum relative error on
[-1/2, 1/2], found with the Remez exchange algorithm (Remez, 1934): solve
for coefficients and the levelled error on n + 2 reference points, move the
points to the extrema of the new error curve, repeat.

Run: python fit_exp2_poly.py   (numpy only)
"""

import numpy as np


def remez_exp2(degree: int, a: float = -0.5, b: float = 0.5, iters: int = 30):
    f = lambda x: np.exp2(x)
    k = np.arange(degree + 2)
    x = (a + b) / 2 + (b - a) / 2 * np.cos(np.pi * k[::-1] / (degree + 1))
    grid = np.linspace(a, b, 200001)
    for _ in range(iters):
        A = np.zeros((degree + 2, degree + 2))
        for i, xi in enumerate(x):
            A[i, : degree + 1] = xi ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1) ** i) * f(xi)
        sol = np.linalg.solve(A, f(x))
        c = sol[: degree + 1]
        err = (np.polyval(c[::-1], grid) - f(grid)) / f(grid)
        segs = np.split(np.arange(grid.size), np.where(np.diff(np.sign(err)) != 0)[0] + 1)
        ext = [s[np.argmax(np.abs(err[s]))] for s in segs]
        if len(ext) > degree + 2:
            ext = sorted(sorted(ext, key=lambda i: -abs(err[i]))[: degree + 2])
        if len(ext) == degree + 2:
            x = grid[ext]
    return c, float(np.abs(err).max())


if __name__ == "__main__":
    c, e = remez_exp2(3)
    c32 = c.astype(np.float32)
    xs = np.linspace(-0.5, 0.5, 100001).astype(np.float32)
    p = np.zeros_like(xs)
    for ci in c32[::-1]:
        p = (p * xs + ci).astype(np.float32)
    rel = np.abs(p.astype(np.float64) - np.exp2(xs.astype(np.float64))) / np.exp2(xs.astype(np.float64))
    print("coefficients c0..c3:", ", ".join(f"{v:.9e}f" for v in c32))
    print(f"max relative error: {e:.3e} (float64), {rel.max():.3e} (float32 Horner)")
