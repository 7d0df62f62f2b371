"""fp64 reference for the attention backward pass (test infrastructure).

The gradient of O = softmax(S) V, S = scale * Q K^T (masked entries -inf),
with respect to Q, K, V for an upstream gradient dO -- the textbook
derivative, written out per (batch, head) in the order the five products of
"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling", §3.2 use (S, then dP = dO V^T, dV = P^T dO,
dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q):

    P      = softmax(S)                     rows; masked keys get P = 0
    D_i    = sum_e dO[i,e] O[i,e]            (= sum_j P_ij dP_ij)
    dV     = P^T dO
    dP     = dO V^T
    dS     = P o (dP - D)
    dQ     = scale * dS K
    dK     = scale * dS^T Q

GQA: a kv head's dK, dV sum the contributions of the query heads that read
it (h // (Hq / Hkv) == g). Causal mask bottom-right: key j visible to query
i iff j <= i + (Sk - Sq). A query row with no visible key contributes 0.

numpy fp64 with the matrix products as library steps; BF16 inputs are
widened exactly.
"""
from __future__ import annotations

from typing import Dict

import numpy as np
import torch


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def attention_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, do: torch.Tensor,
                  scale: float, causal: bool) -> Dict[str, np.ndarray]:
    """dq [B,Sq,Hq,d], dk, dv [B,Sk,Hkv,d] plus o, lse [B,Hq,Sq], delta [B,Hq,Sq]."""
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Sq, Hq, d = qf.shape
    Sk, Hkv = kf.shape[1], kf.shape[2]
    group = Hq // Hkv
    rows = np.arange(Sq)
    keys = np.arange(Sk)
    vis = keys[None, :] <= rows[:, None] + (Sk - Sq) if causal else np.ones((Sq, Sk), bool)
    out = {name: np.zeros(shape) for name, shape in
           (("dq", (B, Sq, Hq, d)), ("dk", (B, Sk, Hkv, d)), ("dv", (B, Sk, Hkv, d)),
            ("o", (B, Sq, Hq, d)), ("lse", (B, Hq, Sq)), ("delta", (B, Hq, Sq)))}
    for b in range(B):
        for h in range(Hq):
            g = h // group
            Q, K, V, dO = qf[b, :, h, :], kf[b, :, g, :], vf[b, :, g, :], dof[b, :, h, :]
            S = np.where(vis, scale * (Q @ K.T), -np.inf)
            m = S.max(axis=1)
            ok = np.isfinite(m)
            E = np.where(vis & ok[:, None], np.exp(S - np.where(ok, m, 0.0)[:, None]), 0.0)
            l = E.sum(axis=1)
            P = np.where(ok[:, None], E / np.where(ok, l, 1.0)[:, None], 0.0)
            O = P @ V
            Dl = (dO * O).sum(axis=1)
            dV = P.T @ dO
            dP = dO @ V.T
            dS = P * (dP - Dl[:, None])
            out["dq"][b, :, h, :] = scale * (dS @ K)
            out["dk"][b, :, g, :] += scale * (dS.T @ Q)
            out["dv"][b, :, g, :] += dV
            out["o"][b, :, h, :] = O
            out["lse"][b, h, :] = np.where(ok, m + np.log(np.where(ok, l, 1.0)), -np.inf)
            out["delta"][b, h, :] = Dl
    return out
