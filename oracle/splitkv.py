"""fp64 model of the key-range split forward and its combine step.

TEST INFRASTRUCTURE (see ``oracle/__init__``). Two functions, each the
plain definition it names:

* ``keyrange_fwd``: attention forward restricted to the keys [k0, k1) --
  the definition of ``ref_attn.c`` with the key sum limited to that range
  (the causal rule still uses the absolute key index: key j is visible to
  query i iff j <= i + (Sk - Sq)). Rows with no visible key in the range get
  O = 0 and LSE = -inf.
* ``merge``: the combine of partial results over disjoint key ranges,
  LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s. This is the
  softmax over a union of disjoint key sets written out; the pages state
  the property it rests on (the output is recovered exactly by the final
  normalisation: "FlashAttention-4: Algorithm and Kernel Pipelining
  Co-Design for Asymmetric Hardware Scaling", Method, §3.1.4).

Plain numpy in fp64, loops over (b, h) only, for small inputs.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np
import torch


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def keyrange_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float, causal: bool,
                 k0: int, k1: int) -> Tuple[np.ndarray, np.ndarray]:
    """O [B,Sq,Hq,d] and LSE [B,Hq,Sq] over the keys k0 <= j < k1 only."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = qf.shape
    Sk, Hkv = kf.shape[1], kf.shape[2]
    group = Hq // Hkv
    k0, k1 = max(0, k0), min(Sk, k1)
    o = np.zeros((B, Sq, Hq, d))
    lse = np.full((B, Hq, Sq), -np.inf)
    if k1 <= k0:
        return o, lse
    keys = np.arange(k0, k1)
    rows = np.arange(Sq)
    visible = (keys[None, :] <= rows[:, None] + (Sk - Sq)) if causal else np.ones((Sq, k1 - k0), bool)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            x = scale * (qf[b, :, h, :] @ kf[b, k0:k1, g, :].T)
            x = np.where(visible, x, -np.inf)
            m = x.max(axis=1)
            ok = np.isfinite(m)
            w = np.where(visible & ok[:, None], np.exp(x - np.where(ok, m, 0.0)[:, None]), 0.0)
            l = w.sum(axis=1)
            num = w @ vf[b, k0:k1, g, :]
            o[b, :, h, :] = np.where(ok[:, None], num / np.where(ok, l, 1.0)[:, None], 0.0)
            lse[b, h, :] = np.where(ok, m + np.log(np.where(ok, l, 1.0)), -np.inf)
    return o, lse


def merge(o_parts: Sequence[np.ndarray], lse_parts: Sequence[np.ndarray]
          ) -> Tuple[np.ndarray, np.ndarray]:
    """Combine partial (O_s [B,Sq,Hq,d], LSE_s [B,Hq,Sq]) over disjoint key ranges."""
    lse_s = np.stack(lse_parts)                          # [S, B, Hq, Sq]
    m = lse_s.max(axis=0)
    ok = np.isfinite(m)
    with np.errstate(invalid="ignore"):
        wts = np.where(ok[None], np.exp(lse_s - np.where(ok, m, 0.0)[None]), 0.0)
    tot = wts.sum(axis=0)
    lse = np.where(ok, m + np.log(np.where(ok, tot, 1.0)), -np.inf)
    o = np.zeros_like(o_parts[0])
    for w_s, o_s in zip(wts, o_parts):
        frac = np.where(ok, w_s / np.where(ok, tot, 1.0), 0.0)   # [B, Hq, Sq]
        o = o + frac.transpose(0, 2, 1)[..., None] * o_s
    return o, lse


def split_ranges(Sk: int, num_splits: int, block: int = 128) -> List[Tuple[int, int]]:
    """The key ranges the split forward uses: whole 128-key blocks,
    ceil(n_blocks / num_splits) per range, empty trailing ranges dropped."""
    nblk = (Sk + block - 1) // block
    per = max(1, (nblk + num_splits - 1) // num_splits)
    out = []
    for s in range(num_splits):
        b0 = s * per
        if b0 >= nblk:
            break
        out.append((b0 * block, min(Sk, (b0 + per) * block)))
    return out
