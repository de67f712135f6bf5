"""Coefficients of the degree-3 polynomial for 2^f, f in [-1/2, 1/2], used by
exp2_poly_x2 in common.cuh: a Remez exchange on the relative error.

Run: python exp2_poly_fit.py  (prints the coefficients c0..c3 and the error)."""
import numpy as np


def remez(n, iters=30, a=-0.5, b=0.5):
    k = np.arange(n + 2)
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * k[::-1] / (n + 1))
    grid = np.linspace(a, b, 200001)
    for _ in range(iters):
        A = np.zeros((n + 2, n + 2))
        for i in range(n + 2):
            A[i, :n + 1] = x[i] ** np.arange(n + 1)
            A[i, n + 1] = -((-1) ** i) * 2 ** x[i]
        c = np.linalg.solve(A, 2 ** x)[:n + 1]
        err = (np.polyval(c[::-1], grid) - 2 ** grid) / 2 ** grid
        cut = np.concatenate([[0], np.where(np.diff(np.sign(err)) != 0)[0] + 1, [len(grid)]])
        ext = [lo + int(np.argmax(np.abs(err[lo:hi]))) for lo, hi in zip(cut[:-1], cut[1:])]
        if len(ext) == n + 2:
            x = grid[ext]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez(3)
    print("c0..c3 =", [float(np.float32(v)) for v in c], "max relative error %.3e" % e)
