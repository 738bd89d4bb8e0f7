"""Fit the cubic used for the FMA-pipe exponential: p(f) ~= 2**f on [0, 1).

Method: minimax fit of the RELATIVE error by the Remez exchange algorithm
(alternation on n+2 points; textbook, e.g. Cheney, "Introduction to
Approximation Theory", ch. 3), with p(0) = 1 imposed so that exact powers of
two stay exact. Run this file to print the coefficients that exp2_poly() in
fa_fwd.cuh uses, in float32, with the maximum relative error over a dense grid.
"""
import numpy as np


def remez_rel(deg=3, iters=30):
    # unknowns: c1..c_deg and E; p(f) = 1 + c1 f + ... ; error e(f) = (p(f) - 2^f) / 2^f
    n = deg  # free coefficients
    x = 0.5 - 0.5 * np.cos(np.pi * np.arange(n + 1) / n)  # n+1 reference points in [0,1]
    x = np.clip(x, 1e-6, 1.0)
    grid = np.linspace(0.0, 1.0, 200001)
    for _ in range(iters):
        A = np.zeros((n + 1, n + 1))
        b = np.zeros(n + 1)
        for i, xi in enumerate(x):
            t = 2.0 ** xi
            A[i, :n] = [xi ** (k + 1) / t for k in range(n)]
            A[i, n] = (-1.0) ** i
            b[i] = 1.0 - 1.0 / t
        sol = np.linalg.solve(A, b)
        c = np.concatenate([[1.0], sol[:n]])
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: extrema of err between sign changes (include the right end)
        idx = [i for i in range(1, len(grid) - 1) if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0]
        idx = [i for i in idx if abs(err[i]) > 0.5 * abs(err).max()] + [len(grid) - 1]
        # keep n+1 alternating extrema
        pts = []
        for i in idx:
            if pts and np.sign(err[i]) == np.sign(err[pts[-1]]):
                if abs(err[i]) > abs(err[pts[-1]]):
                    pts[-1] = i
            else:
                pts.append(i)
        if len(pts) >= n + 1:
            x = grid[pts[-(n + 1):]]
    return c, np.abs(err).max()


if __name__ == "__main__":
    c, e = remez_rel()
    c32 = c.astype(np.float32)
    f = np.linspace(0, 1, 1 << 20, endpoint=False).astype(np.float32)
    p = c32[0] + f * (c32[1] + f * (c32[2] + f * c32[3]))
    rel = np.abs(p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1).max()
    for i, ci in enumerate(c32):
        print(f"c{i} = {float(ci)!r}f  ({ci.view(np.uint32):#010x})")
    print("max relative error (float64 model):", e, " (float32 Horner on grid):", rel)
