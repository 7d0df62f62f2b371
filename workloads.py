"""Seeded synthetic inputs for the attention forward pass.

This module only draws random tensors and names workload shapes. It holds
none of the attention arithmetic, so both the fp64 oracle (test
infrastructure) and the CUDA path can consume the same bytes without sharing
any of the method's code.

Workloads follow the shapes the FlashAttention-4 pages benchmark: BF16
Q/K/V in the [B, S, H, d] layout, head dim 64 or 128, causal and
non-causal, and a GQA case whose row maxima keep rising so the conditional
rescale (threshold tau = 8 in log2 units) actually fires.

Recipe (same for every workload): ``torch.Generator().manual_seed(seed)``,
draws in the order Q, K, V (then the GQA direction q_hat), each ``randn`` in
fp32 and then rounded to BF16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    # GQA stress: K rows get a bias ramp of ``ramp * j * q_hat`` (j = key index).
    ramp: float = 0.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*Hq*Sq*Sk*d, halved when causal (Sq == Sk)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.d
        return f / 2.0 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V, O in BF16 once each, LSE in fp32."""
        q = self.B * self.Sq * self.Hq * self.d * 2
        kv = 2 * self.B * self.Sk * self.Hkv * self.d * 2
        o = q
        lse = self.B * self.Hq * self.Sq * 4
        return q + kv + o + lse

    @property
    def hbm_bytes_fp8(self) -> int:
        """Algorithmic HBM bytes of the FP8 forward: Q, K, V in one byte per
        element, O in BF16, LSE in fp32."""
        in_bf16 = (self.B * self.Sq * self.Hq + 2 * self.B * self.Sk * self.Hkv) * self.d * 2
        return self.hbm_bytes - in_bf16 // 2

    @property
    def hbm_bytes_bwd(self) -> int:
        """Algorithmic HBM bytes of the backward: Q, K, V, O, dO read and dQ,
        dK, dV written in BF16, LSE read in fp32."""
        q = self.B * self.Sq * self.Hq * self.d * 2
        kv = self.B * self.Sk * self.Hkv * self.d * 2
        lse = self.B * self.Hq * self.Sq * 4
        return 3 * q + 2 * kv + lse + q + 2 * kv

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
            "Sq": self.Sq, "Sk": self.Sk, "d": self.d, "causal": self.causal,
            "scale": "1/sqrt(d)", "dtype_in": "bf16",
        }


TINY = Workload("tiny_fwd_b1_h2_s256_d64", 1, 2, 2, 256, 256, 64, False)
MID = Workload("mid_fwd_b4_h16_s2048_d128", 4, 16, 16, 2048, 2048, 128, False)
LONG_CAUSAL = Workload("long_causal_fwd_b2_h16_s8192_d128", 2, 16, 16, 8192, 8192, 128, True)
GQA_STRESS = Workload("gqa_causal_stress_b1_hq32_hkv8_s16384_d128", 1, 32, 8, 16384, 16384, 128,
                      True, ramp=0.002)


def d64_sweep() -> List[Workload]:
    """Head-dim-64 sweep: Hq = Hkv = 32, B*S = 32768 tokens, both masks."""
    out = []
    for S in (1024, 4096, 16384, 32768):
        B = 32768 // S
        for causal in (False, True):
            tag = "causal" if causal else "noncausal"
            out.append(Workload(f"d64_{tag}_b{B}_h32_s{S}", B, 32, 32, S, S, 64, causal))
    return out


ALL_NAMED = [TINY, MID, LONG_CAUSAL, GQA_STRESS] + d64_sweep()

# Few query tiles, many keys: 4 query-tile pairs per head x 16 heads = 64
# work tiles on 152 SMs -- the shape the key-range split forward is for.
SPLIT_LONG_KEYS = Workload("splitkv_fwd_b1_h16_sq1024_sk65536_d128", 1, 16, 16, 1024, 65536, 128,
                           False)
EXTRA = [SPLIT_LONG_KEYS]


def by_name(name: str) -> Workload:
    for w in ALL_NAMED + EXTRA:
        if w.name == name:
            return w
    raise KeyError(name)


def make_inputs(w: Workload, seed: int = 0, *, batch_offset: int = 0
                ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Return BF16 CPU tensors q [B,Sq,Hq,d], k, v [B,Sk,Hkv,d].

    ``batch_offset`` shifts the seed so that shards of a larger global batch
    (one per rank) draw distinct data.
    """
    g = torch.Generator().manual_seed(seed + 1000003 * batch_offset)
    q = torch.randn((w.B, w.Sq, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    if w.ramp != 0.0:
        q_hat = torch.randn((w.d,), generator=g, dtype=torch.float32)
        q_hat = q_hat / q_hat.norm()
        j = torch.arange(w.Sk, dtype=torch.float32).view(1, w.Sk, 1, 1)
        k = k + w.ramp * j * q_hat.view(1, 1, 1, w.d)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


E4M3_MAX = 448.0   # largest finite e4m3 value


def quantize_e4m3(x: torch.Tensor) -> Tuple[torch.Tensor, float]:
    """Per-tensor e4m3 quantisation of an fp32/BF16 tensor for FP8 inputs.

    scale = amax / 448 (amax = largest |x|); codes = round-to-nearest-even
    of x / scale in torch's float8_e4m3fn conversion. Returns (codes, scale)
    with x ~ codes * scale.
    """
    x = x.to(torch.float32)
    amax = float(x.abs().max()) if x.numel() else 0.0
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    codes = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes, scale


def make_inputs_fp8(w: Workload, seed: int = 0, *, batch_offset: int = 0):
    """FP8 inputs of a head-dim-128 workload: the fp32 draws of
    ``make_inputs`` (same seed, same order), each tensor quantised with
    ``quantize_e4m3``. Returns (q8, k8, v8, q_scale, k_scale, v_scale)."""
    g = torch.Generator().manual_seed(seed + 1000003 * batch_offset)
    q = torch.randn((w.B, w.Sq, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    if w.ramp != 0.0:
        q_hat = torch.randn((w.d,), generator=g, dtype=torch.float32)
        q_hat = q_hat / q_hat.norm()
        j = torch.arange(w.Sk, dtype=torch.float32).view(1, w.Sk, 1, 1)
        k = k + w.ramp * j * q_hat.view(1, 1, 1, w.d)
    (q8, qs), (k8, ks), (v8, vs) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    return q8, k8, v8, qs, ks, vs


def make_custom_fp8(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int = 128, seed: int = 0,
                    dist: str = "randn"):
    """Seeded FP8 inputs of arbitrary shape: ``make_custom``'s draws (before
    the BF16 rounding) quantised per tensor. Same return as make_inputs_fp8."""
    g = torch.Generator().manual_seed(seed)
    mul = 4.0 if dist == "wide" else 1.0
    if dist not in ("randn", "wide"):
        raise ValueError(dist)
    q = mul * torch.randn((B, Sq, Hq, d), generator=g)
    k = mul * torch.randn((B, Sk, Hkv, d), generator=g)
    v = torch.randn((B, Sk, Hkv, d), generator=g)
    (q8, qs), (k8, ks), (v8, vs) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    return q8, k8, v8, qs, ks, vs


def make_custom(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int, seed: int = 0,
                dist: str = "randn") -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Seeded BF16 inputs of arbitrary shape for edge-case tests."""
    g = torch.Generator().manual_seed(seed)
    shape_q = (B, Sq, Hq, d)
    shape_kv = (B, Sk, Hkv, d)
    if dist == "randn":
        q = torch.randn(shape_q, generator=g)
        k = torch.randn(shape_kv, generator=g)
        v = torch.randn(shape_kv, generator=g)
    elif dist == "wide":  # large-magnitude logits: stresses max tracking
        q = 4.0 * torch.randn(shape_q, generator=g)
        k = 4.0 * torch.randn(shape_kv, generator=g)
        v = torch.randn(shape_kv, generator=g)
    else:
        raise ValueError(dist)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def sample_rows(w: Workload, n_random: int, seed: int = 0, edge: int = 128,
                max_bh: Optional[int] = None) -> torch.Tensor:
    """Deterministic row subset for full-size checks and the CPU baseline.

    Returns int64 flat row ids ``(b*Hq + h)*Sq + i``: for each (b, h) (or the
    first ``max_bh`` of them) the first and last ``edge`` rows, plus
    ``n_random`` seeded random rows over the whole output.
    """
    g = torch.Generator().manual_seed(seed + 7)
    n_bh = w.B * w.Hq
    bhs = range(n_bh if max_bh is None else min(n_bh, max_bh))
    ids = []
    e = min(edge, w.Sq)
    for bh in bhs:
        base = bh * w.Sq
        ids.append(torch.arange(base, base + e))
        ids.append(torch.arange(base + w.Sq - e, base + w.Sq))
    if n_random > 0:
        ids.append(torch.randint(0, n_bh * w.Sq, (n_random,), generator=g))
    return torch.unique(torch.cat(ids)).to(torch.int64)
