"""ctypes front end of the fp64 C reference (test infrastructure).

The C file computes the plain definition of attention forward (see the
header of ``ref_attn.c``; "FlashAttention-4: Algorithm and Kernel
Pipelining Co-Design for Asymmetric Hardware Scaling", Method and §3.1.4:
the final 1/l normalisation gives the exact softmax-times-V output).
Inputs are BF16 torch tensors (their bit patterns are widened exactly);
outputs are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np
import torch

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                        dbl, ctypes.c_int]
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_fwd_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl,
                                             ctypes.c_int, vp, i64, vp, vp]
        lib.oracle_attn_fwd_rows.restype = ctypes.c_int
        lib.oracle_attn_probs.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl,
                                          ctypes.c_int, i64, i64, vp]
        lib.oracle_attn_probs.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype != torch.bfloat16:
        raise TypeError("oracle inputs are BF16 tensors")
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()
                                ).view(np.uint16)


def _shape(q, k, v):
    B, Sq, Hq, d = q.shape
    Bk, Sk, Hkv, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch")
    return B, Sq, Hq, Hkv, Sk, d


def attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                  causal: bool) -> Tuple[np.ndarray, np.ndarray]:
    """Full output: O [B,Sq,Hq,d] fp64 and LSE [B,Hq,Sq] fp64."""
    B, Sq, Hq, Hkv, Sk, d = _shape(q, k, v)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    o = np.zeros((B, Sq, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, Sq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                 o.ctypes.data, lse.ctypes.data, B, Hq, Hkv, Sq, Sk, d,
                                 float(scale), int(bool(causal)))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (rc={rc})")
    return o, lse


def attention_fwd_rows(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                       causal: bool, rows) -> Tuple[np.ndarray, np.ndarray]:
    """Only the listed flat rows ``(b*Hq + h)*Sq + i``: O [n, d], LSE [n]."""
    B, Sq, Hq, Hkv, Sk, d = _shape(q, k, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    o = np.zeros((rows.size, d), dtype=np.float64)
    lse = np.zeros((rows.size,), dtype=np.float64)
    rc = _load().oracle_attn_fwd_rows(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                      B, Hq, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                                      rows.ctypes.data, rows.size, o.ctypes.data,
                                      lse.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_rows rejected its arguments (rc={rc})")
    return o, lse


def attention_probs(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                    causal: bool, b: int = 0, h: int = 0) -> np.ndarray:
    """Softmax matrix P [Sq, Sk] of one (b, h)."""
    B, Sq, Hq, Hkv, Sk, d = _shape(q, k, v)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    p = np.zeros((Sq, Sk), dtype=np.float64)
    rc = _load().oracle_attn_probs(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                   B, Hq, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                                   int(b), int(h), p.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_attn_probs rejected its arguments (rc={rc})")
    return p


def gather_rows(o_full: np.ndarray, lse_full: np.ndarray, rows, Hq: int, Sq: int
                ) -> Tuple[np.ndarray, np.ndarray]:
    """Pick flat rows out of full [B,Sq,Hq,d] / [B,Hq,Sq] arrays."""
    rows = np.asarray(rows, dtype=np.int64)
    i = rows % Sq
    h = (rows // Sq) % Hq
    b = rows // (Sq * Hq)
    return o_full[b, i, h, :], lse_full[b, h, i]
