"""fp64 model of the tile-by-tile online softmax with conditional rescale.

TEST INFRASTRUCTURE (see ``oracle/__init__``). It follows the algebra of
"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling", Method and §3.1.4 (Eq. 6), in the pages' order:

  * logits live in the log2 domain: t_ij = c * (q_i . k_j), c = scale*log2(e);
  * keys are visited in blocks of ``block_n`` (128 on the pages' tiles);
  * per row a reference max m~ and a running sum l are kept; the rescale
    (alpha = 2^(m~ - m_new), applied to l and O) is skipped while the new
    block max exceeds m~ by no more than tau (tau = log2 256 = 8 on the
    pages; tau = 0 is the classic eager online softmax);
  * the decision is taken per group of ``gate_rows`` rows ("warp
    granularity"): if any row in the group needs it, every row in the group
    moves to its own exact new max;
  * p = 2^(t - m~); the final O / l and LSE = ln2 * (m~ + log2 l) recover
    the exact result.

The exact definition lives in ``ref_attn.c``; this model exists to check
that the conditional rescale is exact algebra (it must equal the definition
to fp64 rounding for every tau) and to count how many rescales it skips.
Reading taken where the pages are silent: the new block max is compared
with the reference max m~ used for the last rescale (not the previous
block's max), so p never exceeds 2^tau.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np
import torch

LOG2E = 1.0 / math.log(2.0)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def tiled_attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                        causal: bool, tau: float = 8.0, block_n: int = 128,
                        gate_rows: int = 32) -> Tuple[np.ndarray, np.ndarray, dict]:
    """Return O [B,Sq,Hq,d], LSE [B,Hq,Sq] (fp64) and rescale statistics."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = qf.shape
    Sk, Hkv = kf.shape[1], kf.shape[2]
    group = Hq // Hkv
    c = scale * LOG2E
    o_out = np.zeros((B, Sq, Hq, d))
    lse_out = np.zeros((B, Hq, Sq))
    n_rescale_groups = 0       # (row group, block) pairs that rescaled after block 0
    n_group_blocks = 0         # (row group, block) pairs visited after block 0
    rows = np.arange(Sq)
    n_groups = (Sq + gate_rows - 1) // gate_rows
    for b in range(B):
        for h in range(Hq):
            g = h // group
            qh = qf[b, :, h, :]                # [Sq, d]
            kh = kf[b, :, g, :]                # [Sk, d]
            vh = vf[b, :, g, :]
            m_ref = np.full(Sq, -np.inf)
            l = np.zeros(Sq)
            o = np.zeros((Sq, d))
            for j0 in range(0, Sk, block_n):
                cols = np.arange(j0, min(j0 + block_n, Sk))
                t = c * (qh @ kh[cols].T)      # [Sq, n] log2-domain logits
                if causal:
                    allowed = cols[None, :] <= rows[:, None] + (Sk - Sq)
                    t = np.where(allowed, t, -np.inf)
                m_blk = t.max(axis=1)
                m_new = np.maximum(m_ref, m_blk)
                with np.errstate(invalid="ignore"):
                    need = m_new > m_ref + tau          # -inf + tau stays -inf
                need_pad = np.zeros(n_groups * gate_rows, dtype=bool)
                need_pad[:Sq] = need
                need_grp = need_pad.reshape(n_groups, gate_rows).any(axis=1)
                gate = np.repeat(need_grp, gate_rows)[:Sq]
                if j0 > 0:
                    n_group_blocks += n_groups
                    n_rescale_groups += int(need_grp.sum())
                move = gate & np.isfinite(m_new)
                alpha = np.ones(Sq)
                with np.errstate(invalid="ignore"):
                    alpha[move] = np.exp2(m_ref[move] - m_new[move])   # 0 when m_ref = -inf
                l = l * alpha
                o = o * alpha[:, None]
                m_ref = np.where(move, m_new, m_ref)
                m_use = np.where(np.isfinite(m_ref), m_ref, 0.0)
                p = np.exp2(t - m_use[:, None])       # exp2(-inf) = 0 for masked keys
                l = l + p.sum(axis=1)
                o = o + p @ vh[cols]
            with np.errstate(divide="ignore", invalid="ignore"):
                o_fin = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
                lse = np.where(l > 0, (m_ref + np.log2(np.where(l > 0, l, 1.0))) / LOG2E,
                               -np.inf)
            o_out[b, :, h, :] = o_fin
            lse_out[b, h, :] = lse
    stats = {"rescaled_group_blocks": n_rescale_groups, "group_blocks": n_group_blocks}
    return o_out, lse_out, stats
