"""Model of the software 2^x used beside MUFU.EX2 (test infrastructure).

Follows "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", §3.1.3 and Table 2: 2^x = 2^floor(x) *
2^frac(x); the integer part goes into the IEEE-754 exponent field by
integer arithmetic, the fractional part is a polynomial evaluated by
Horner's rule on FMA units. The pages use a Sollya-tuned polynomial whose
coefficients they do not print; this module fits its own.

Fit (this file's own method): minimax RELATIVE error of
p(f) = 1 + c1 f + ... + cn f^n against 2^f on [0, 1], with p(0) = 1 held
exact, solved as a linear program on a dense grid (discretised minimax,
``scipy.optimize.linprog``). Coefficients are then rounded to fp32, the
precision the kernel evaluates in.

Reading where the pages are silent: inputs are clamped to x >= -127, so
the result for x <= -127 is a value below 2^-126 (it plays the role of the
hardware's flush to zero: no softmax entry that small matters).
"""
from __future__ import annotations

import functools
from typing import Tuple

import numpy as np


@functools.lru_cache(maxsize=None)
def fit_minimax(degree: int = 3, n_grid: int = 4097) -> Tuple[Tuple[float, ...], float]:
    """Return ((c1..cn) in fp64, max relative error) of the LP minimax fit."""
    from scipy.optimize import linprog

    f = np.linspace(0.0, 1.0, n_grid)
    target = np.exp2(f)
    # variables: c1..cn, E ; minimise E
    # (1 + sum c_k f^k) / 2^f - 1 <= E   and  >= -E
    powers = np.stack([f ** k for k in range(1, degree + 1)], axis=1) / target[:, None]
    resid0 = 1.0 / target - 1.0
    ones = np.ones((n_grid, 1))
    a_ub = np.vstack([np.hstack([powers, -ones]), np.hstack([-powers, -ones])])
    b_ub = np.concatenate([-resid0, resid0])
    cost = np.zeros(degree + 1)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1),
                  method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    coeffs = tuple(float(x) for x in res.x[:degree])
    return coeffs, float(res.x[degree])


def coeffs_f32(degree: int = 3) -> np.ndarray:
    c, _ = fit_minimax(degree)
    return np.asarray(c, dtype=np.float32)


def poly_f32(frac: np.ndarray, coeffs: np.ndarray) -> np.ndarray:
    """Horner in fp32, one rounding per step: 1 + f(c1 + f(c2 + f c3))."""
    frac = frac.astype(np.float32)
    acc = np.full_like(frac, coeffs[-1], dtype=np.float32)
    for c in coeffs[-2::-1]:
        acc = (acc * frac + np.float32(c)).astype(np.float32)
    return (acc * frac + np.float32(1.0)).astype(np.float32)


def exp2_emulated(x: np.ndarray, degree: int = 3) -> np.ndarray:
    """Cody-Waite range reduction + polynomial, fp32 in and out."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-127.0))
    n = np.floor(x).astype(np.float32)
    frac = (x - n).astype(np.float32)              # exact in fp32, in [0, 1)
    p = poly_f32(frac, coeffs_f32(degree))
    bits = p.view(np.int32) + (n.astype(np.int32) << 23)   # add n to the exponent field
    return bits.astype(np.int32).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest BF16 (ties to even); returns fp32 values."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|bit distance| between non-negative BF16-representable fp32 values."""
    ia = (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.int64)
    ib = (np.asarray(b, np.float32).view(np.uint32) >> 16).astype(np.int64)
    return np.abs(ia - ib)


def bf16_grid(lo: float, hi: float) -> np.ndarray:
    """Every finite BF16 value in [lo, hi], as fp32, sorted ascending."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    vals = vals[(vals >= lo) & (vals <= hi)]
    return np.unique(vals)
