"""fp64 oracle of the FP8 (e4m3) attention forward (test infrastructure).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may use this module; the product
never does.

"How FlashAttention 4 Works", the section on which steps may run in low
precision: Q K^T and P V take FP8 inputs on the tensor cores with an fp32
accumulator, the softmax (max, exponential, sum) stays in fp32 and the
output is stored in BF16. The inputs are e4m3 codes with one dequantisation
scale per tensor, so the quantity computed is the ordinary attention
forward ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", Method) of the true values
    Q = q_scale q8,  K = k_scale k8,  V = v_scale v8:
    S = scale Q K^T [bottom-right causal mask],  P = softmax(S),
    O = P V,  LSE = logsumexp(S) per row.

The e4m3 code is read by its definition (OCP 8-bit floating point, E4M3):
sign bit 7, a 4-bit exponent with bias 7 in bits 6-3, a 3-bit mantissa in
bits 2-0; exponent 0 is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7
is NaN; there are no infinities, so the largest finite value is 448.

The bound returned beside O is the part of the error the method adds when
P, an fp32 value, is rounded to e4m3 before the P V product: with three
mantissa bits, round-to-nearest moves a normal value by at most 2^-4 of
itself, and a value below the smallest normal 2^-6 by at most half the
subnormal spacing, 2^-10, and never by more than itself (it can only fall
to zero). The kernel's P is the true P times 2^c with c >= 0 (the row
maximum it subtracts may be stale by up to the rescale threshold), so in
true units the error of P_ij is at most
    e_ij = max(P_ij / 16, min(P_ij, 2^-10)),  P_ij = exp(S_ij - max_j S_ij) <= 1;
summing over keys against |V| and dividing by the row sum l_i bounds the
error of O:
    bound_ic = sum_j e_ij |V_jc| / l_i.
That worst case adds every key's error with the same sign. Round-to-nearest
errors of different keys are close to independent, each at most the term
above, so the root-sum-square
    rss_ic = sqrt(sum_j (e_ij V_jc)^2) / l_i
is the scale the actual error has (for long rows far below the bound).
"""
from __future__ import annotations

from typing import Tuple

import numpy as np
import torch


def e4m3_to_float(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 e4m3 codes to fp64 values by the bit-field definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, out)


def codes_of(t: torch.Tensor) -> np.ndarray:
    """uint8 bit patterns of a float8_e4m3fn (or uint8) tensor."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError("FP8 oracle inputs are float8_e4m3fn or uint8 codes")
    return t.numpy()


def _dequant(t: torch.Tensor, s: float) -> np.ndarray:
    return e4m3_to_float(codes_of(t)) * float(s)


def _rows_fwd(Q, K, V, scale, causal, rows, Hq, Hkv, Sq, Sk, with_bound):
    """Per flat row id (b*Hq + h)*Sq + i: O [n, d], LSE [n], bound, rss [n, d]."""
    rows = np.asarray(rows, dtype=np.int64)
    d = Q.shape[-1]
    group = Hq // Hkv
    o = np.zeros((rows.size, d))
    lse = np.full((rows.size,), -np.inf)
    bound = np.zeros((rows.size, d))
    rss = np.zeros((rows.size, d))
    i_all = rows % Sq
    h_all = (rows // Sq) % Hq
    b_all = rows // (Sq * Hq)
    for n in range(rows.size):
        b, h, i = int(b_all[n]), int(h_all[n]), int(i_all[n])
        hk = h // group
        hi = Sk if not causal else min(Sk, i + (Sk - Sq) + 1)   # keys j <= i + Sk - Sq
        if hi <= 0:
            continue                                          # no visible key: O = 0, LSE = -inf
        s = scale * (K[b, :hi, hk, :] @ Q[b, i, h, :])
        m = s.max()
        p = np.exp(s - m)
        l = p.sum()
        o[n] = (p @ V[b, :hi, hk, :]) / l
        lse[n] = m + np.log(l)
        if with_bound:   # p = exp(S - max) <= 1 per key; O divides by l
            e = np.maximum(p / 16.0, np.minimum(p, 2.0 ** -10))
            bound[n] = (e @ np.abs(V[b, :hi, hk, :])) / l
            rss[n] = np.sqrt((e * e) @ (V[b, :hi, hk, :] ** 2)) / l
    return o, lse, bound, rss


def attention_fwd_fp8_rows(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor,
                           q_scale: float, k_scale: float, v_scale: float, scale: float,
                           causal: bool, rows
                           ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """O [n, d], LSE [n], and the e4m3-P rounding bound and root-sum-square
    [n, d] for flat rows.

    q8 [B, Sq, Hq, d], k8 / v8 [B, Sk, Hkv, d] e4m3 codes; the bound and
    the rss are in the units of O (they include v_scale).
    """
    B, Sq, Hq, d = q8.shape
    _, Sk, Hkv, _ = k8.shape
    Q, K, V = _dequant(q8, q_scale), _dequant(k8, k_scale), _dequant(v8, v_scale)
    return _rows_fwd(Q, K, V, float(scale), bool(causal), rows, Hq, Hkv, Sq, Sk, True)


def attention_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: float,
                      k_scale: float, v_scale: float, scale: float, causal: bool
                      ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Full output: O [B,Sq,Hq,d], LSE [B,Hq,Sq], bound and rss [B,Sq,Hq,d]."""
    B, Sq, Hq, d = q8.shape
    rows = np.arange(B * Hq * Sq, dtype=np.int64)
    o, lse, bound, rss = attention_fwd_fp8_rows(q8, k8, v8, q_scale, k_scale, v_scale, scale,
                                                causal, rows)

    def to_bshd(x):
        return np.ascontiguousarray(x.reshape(B, Hq, Sq, d).transpose(0, 2, 1, 3))

    return to_bshd(o), lse.reshape(B, Hq, Sq), to_bshd(bound), to_bshd(rss)
