"""Fit the cubic used for the FMA-pipe exponential: p(f) ~= 2**f on [0, 1).

Method: minimax fit of the RELATIVE error by the Remez exchange algorithm
(alternation on n+1 points for the n free coefficients; textbook, e.g.
Cheney, "Introduction to Approximation Theory", ch. 3), Two fits are printed, each in float32 with its maximum relative error over a
dense grid:
  [-1/2, 1/2] with all four coefficients free: the one exp2_poly() and
               exp2_poly2() in fa_fwd.cuh use (x = round(x) + f, rounding by
               the 1.5*2^23 trick);
  [0, 1) with p(0) = 1 imposed: the variant for x = floor(x) + f, kept for
               comparison (floor and float-to-int conversions run on the
               transcendental pipe, which the kernel's path avoids).
"""
import numpy as np


def remez_rel(deg=3, iters=30, lo=0.0, hi=1.0, fix0=True):
    # p(f) = c0 + c1 f + ... ; relative error e(f) = (p(f) - 2^f) / 2^f.
    # fix0: c0 = 1 is imposed and c1..c_deg are free; otherwise c0..c_deg are free.
    n = deg if fix0 else deg + 1  # free coefficients
    k0 = 1 if fix0 else 0         # power of the first free coefficient
    x = lo + (hi - lo) * (0.5 - 0.5 * np.cos(np.pi * np.arange(n + 1) / n))  # n+1 reference points
    x = np.where(np.abs(x) < 1e-6, 1e-6, x)
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        A = np.zeros((n + 1, n + 1))
        b = np.zeros(n + 1)
        for i, xi in enumerate(x):
            t = 2.0 ** xi
            A[i, :n] = [xi ** (k + k0) / t for k in range(n)]
            A[i, n] = (-1.0) ** i
            b[i] = (1.0 - 1.0 / t) if fix0 else 1.0
        sol = np.linalg.solve(A, b)
        c = np.concatenate([[1.0], sol[:n]]) if fix0 else sol[:n]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: extrema of err between sign changes (include the right end)
        idx = [i for i in range(1, len(grid) - 1) if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0]
        idx = [0] + [i for i in idx if abs(err[i]) > 0.5 * abs(err).max()] + [len(grid) - 1]
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
    for lo, hi, fix0 in ((0.0, 1.0, True), (-0.5, 0.5, False)):
        c, e = remez_rel(lo=lo, hi=hi, fix0=fix0)
        c32 = c.astype(np.float32)
        f = np.linspace(lo, hi, 1 << 20, endpoint=False).astype(np.float32)
        p = c32[0] + f * (c32[1] + f * (c32[2] + f * c32[3]))
        rel = np.abs(p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1).max()
        print(f"interval [{lo}, {hi}]" + (" with p(0) = 1" if fix0 else " (all coefficients free)"))
        for i, ci in enumerate(c32):
            print(f"  c{i} = {float(ci)!r}f  ({ci.view(np.uint32):#010x})")
        print("  max relative error (float64 model):", e, " (float32 Horner on grid):", rel)
