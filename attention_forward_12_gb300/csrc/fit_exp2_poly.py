"""Fit the polynomial of the kernel's FMA-pipe exp2.

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(Cody and Waite's argument reduction, "Software Manual for the Elementary
Functions", 1980); 2^f is approximated by the polynomial of degree `deg`
that minimises the maximum RELATIVE error on [-1/2, 1/2], found with the
Remez exchange algorithm.  The constant term is pinned to 1 so that
2^0 = 1 exactly.  Run:  python fit_exp2_poly.py [deg]
"""
import sys

import numpy as np


def remez_relative(deg: int, iters: int = 40):
    a, b = -0.5, 0.5
    f = lambda x: np.exp2(x)
    # unknowns: c1..c_deg (c0 = 1) and the levelled error E; deg+1 alternation points
    k = np.arange(deg + 1)
    xs = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * (deg - k) / deg)  # Chebyshev extrema
    for _ in range(iters):
        # (1 + sum c_i x^i) / 2^x - 1 = (-1)^j E at each point
        A = np.zeros((deg + 1, deg + 1))
        rhs = np.zeros(deg + 1)
        for j, x in enumerate(xs):
            A[j, :deg] = [x ** i / f(x) for i in range(1, deg + 1)]
            A[j, deg] = -((-1) ** j)
            rhs[j] = 1.0 - 1.0 / f(x)
        sol = np.linalg.solve(A, rhs)
        c = np.concatenate([[1.0], sol[:deg]])
        grid = np.linspace(a, b, 200001)
        err = np.polyval(c[::-1], grid) / f(grid) - 1.0
        # new alternation points: extrema of err between sign changes
        idx = [0]
        for i in range(1, len(grid) - 1):
            if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0:
                idx.append(i)
        idx.append(len(grid) - 1)
        cand = grid[idx]
        ev = err[idx]
        # keep deg+1 points with alternating signs and largest magnitudes
        pts = []
        for x, e in zip(cand, ev):
            if pts and np.sign(e) == np.sign(pts[-1][1]):
                if abs(e) > abs(pts[-1][1]):
                    pts[-1] = (x, e)
            else:
                pts.append((x, e))
        while len(pts) > deg + 1:
            if abs(pts[0][1]) < abs(pts[-1][1]):
                pts.pop(0)
            else:
                pts.pop()
        if len(pts) == deg + 1:
            xs = np.array([p[0] for p in pts])
    return c, float(np.abs(err).max())


def eval_fp32(c, x):
    """Emulate the kernel in float32: round-to-nearest n via the 1.5*2^23
    shift, f = x - n, Horner in fp32 with fused multiply-add, 2^n applied by
    adding n to the exponent field."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    fr = (x - n).astype(np.float32)
    cf = [np.float32(v) for v in c]
    p = np.full_like(fr, cf[-1])
    for v in cf[-2::-1]:  # fused: one rounding per step
        p = (p.astype(np.float64) * fr.astype(np.float64) + np.float64(v)).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.view(np.float32)


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 4
    c, e = remez_relative(deg)
    print(f"degree {deg}: max relative error {e:.3e} (real arithmetic)")
    for i, v in enumerate(c):
        print(f"  c{i} = {np.float32(v).item()!r}f  // {v!r}")
    xs = np.linspace(-126, 8, 2000001, dtype=np.float32)
    rel = np.abs(eval_fp32(c, xs).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1)
    print(f"fp32 evaluation on [-126, 8]: max relative error {rel.max():.3e}")
