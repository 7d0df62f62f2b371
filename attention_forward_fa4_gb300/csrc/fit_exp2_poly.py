"""Derive the coefficients of the kernel's software 2^x polynomial.

"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling" (§3.1.3, Table 2) computes 2^x = 2^floor(x) * 2^frac on
the FMA units, with the fractional part from a low-degree polynomial
(degree 3 is enough for BF16 outputs). The pages do not print their
coefficients, so this script derives ours:

  p(f) = 1 + c1 f + c2 f^2 + c3 f^3,  f in [0, 1],
  minimising max |p(f) / 2^f - 1|  (relative error), with p(0) = 1 exact,

by the Remez exchange algorithm (levelled error on 4 reference points,
exchange to the extrema of the error curve until they equioscillate).
The fp32-rounded results are the constants in ``fa4_exp2.cuh``.

Run: ``python fit_exp2_poly.py`` (prints the constants and the error).
"""
from __future__ import annotations

import numpy as np


def _error(c, f):
    p = 1.0 + f * (c[0] + f * (c[1] + f * c[2]))
    return p / np.exp2(f) - 1.0


def remez(iters: int = 30, grid: int = 400001):
    ref = np.array([0.1, 0.45, 0.8, 1.0])          # initial reference points
    f = np.linspace(0.0, 1.0, grid)
    c = np.zeros(3)
    for _ in range(iters):
        # Solve  sum_k c_k x^k / 2^x - (-1)^i E = 1 - 1/2^x  at the references.
        inv = np.exp2(-ref)
        a = np.stack([ref * inv, ref ** 2 * inv, ref ** 3 * inv,
                      -((-1.0) ** np.arange(4))], axis=1)
        sol = np.linalg.solve(a, 1.0 - inv)
        c = sol[:3]
        e = _error(c, f)
        # local extrema of the error (interior) plus the right end point
        idx = np.where((np.abs(e[1:-1]) >= np.abs(e[:-2])) &
                       (np.abs(e[1:-1]) >= np.abs(e[2:])))[0] + 1
        idx = np.unique(np.append(idx, grid - 1))
        idx = idx[np.abs(e[idx]) > 0]
        # keep one point per sign run (the largest), need 4 alternations
        runs, cur = [], [idx[0]]
        for i in idx[1:]:
            if np.sign(e[i]) == np.sign(e[cur[-1]]):
                cur.append(i)
            else:
                runs.append(max(cur, key=lambda t: abs(e[t])))
                cur = [i]
        runs.append(max(cur, key=lambda t: abs(e[t])))
        if len(runs) < 4:
            break
        while len(runs) > 4:                         # drop the smallest end
            runs = runs[1:] if abs(e[runs[0]]) < abs(e[runs[-1]]) else runs[:-1]
        ref = f[np.array(runs)]
    return c, float(np.abs(_error(c, f)).max())


if __name__ == "__main__":
    c, err = remez()
    c32 = c.astype(np.float32)
    print("c1..c3 =", ", ".join(f"{x:.9e}f" for x in c32))
    print(f"max relative error = {err:.4e} (2^{np.log2(err):.2f})")
