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
