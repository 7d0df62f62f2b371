"""Comparison helpers shared by the GPU parity tests.

Tolerances (from the target statement of the forward pass): O max-abs
error <= 2e-2 and mean-abs error <= 2e-3 against the fp64 oracle, LSE
max-abs error <= 1e-3. The kernel stores O in BF16 (relative spacing 2^-8)
and rounds P to BF16 before the P*V product, so an |O| of order 1 carries
about 4e-3 of rounding by itself; 2e-2 leaves room for the tails of
|O| ~ 3 rows. LSE is computed in fp32 from fp32 sums.
"""
from __future__ import annotations

import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def errors(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    fin = np.isfinite(lse_ref)
    if not (np.isfinite(lse_gpu) == fin).all():
        raise AssertionError("finite / -inf pattern of LSE differs from the oracle")
    if not (lse_gpu[~fin] == -np.inf).all():
        raise AssertionError("rows without keys must have LSE = -inf")
    eo = np.abs(o_gpu - o_ref)
    el = np.abs(lse_gpu[fin] - lse_ref[fin]) if fin.any() else np.zeros(1)
    return float(eo.max()) if eo.size else 0.0, float(eo.mean()) if eo.size else 0.0, \
        float(el.max())


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what: str = ""):
    mx, mean, lmx = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    msg = f"{what}: O max {mx:.3e} mean {mean:.3e}, LSE max {lmx:.3e}"
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS and lmx <= LSE_MAX_ABS, msg
    return mx, mean, lmx


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def gather_gpu_rows(o: torch.Tensor, lse: torch.Tensor, rows: torch.Tensor):
    """Flat rows (b*Hq + h)*Sq + i of GPU outputs, on the host."""
    B, Sq, Hq, d = o.shape
    rows = rows.to(torch.int64)
    i = rows % Sq
    h = (rows // Sq) % Hq
    b = rows // (Sq * Hq)
    dev = o.device
    o_r = o[b.to(dev), i.to(dev), h.to(dev), :]
    l_r = lse[b.to(dev), h.to(dev), i.to(dev)]
    return to_np(o_r), to_np(l_r)


# FP8 forward: no stated tolerance; derived from the e4m3 rounding of P (see
# oracle/fp8.py for `bound` and `rss`) plus the BF16 rounding of O
# (half a BF16 ulp = 2^-8 relative) and an fp32-accumulation floor.
FP8_ABS_FLOOR = 1e-4
FP8_RSS_RATIO = 1.0


def assert_close_fp8(o_gpu, lse_gpu, o_ref, lse_ref, bound, rss, what: str = ""):
    """Element-wise worst case, a root-mean-square check against the rss
    scale, and the LSE check of the BF16 path."""
    mx, mean, lmx = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    err = np.abs(np.asarray(o_gpu, dtype=np.float64) - o_ref)
    out_round = 2.0 ** -8 * np.abs(o_ref)
    worst = bound + out_round + FP8_ABS_FLOOR
    over = float((err / worst).max()) if err.size else 0.0
    ratio = float(np.sqrt(np.mean((err / (rss + out_round + 1e-6)) ** 2))) if err.size else 0.0
    msg = (f"{what}: O max {mx:.3e} mean {mean:.3e} (worst-case use {over:.3f}, "
           f"rms/rss {ratio:.3f}), LSE max {lmx:.3e}")
    assert over <= 1.0 and ratio <= FP8_RSS_RATIO and lmx <= LSE_MAX_ABS, msg
    return mx, mean, lmx, over, ratio
