"""Pins of the oracle's BF16 helpers (``oracle/exp2_emu.py``: ``bf16_round``,
``bf16_ulp_distance``), which decide the Table 2 accuracy statistic of
"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling", §3.1.3 (degree-3 2^x within 1 BF16 ULP on 99 % of
inputs).

Both helpers work on fp32 bit patterns. They are checked here against
torch's own fp32 -> bfloat16 conversion (round to nearest, ties to even)
and against ``torch.nextafter`` on bfloat16, which share none of their
arithmetic.
"""
import numpy as np
import torch

from oracle import exp2_emu as e

# Low halves of the fp32 pattern that decide the rounding: exact, just above
# zero, just below / at / just above the half-way tie, and the largest.
_LOW = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFE, 0xFFFF],
                dtype=np.uint32)


def _patterns(seed: int = 5) -> np.ndarray:
    """Every upper half (all signs, exponents incl. subnormals, mantissas)
    combined with the critical low halves, plus seeded random patterns."""
    hi = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    bits = (hi[:, None] | _LOW[None, :]).ravel()
    rnd = np.random.default_rng(seed).integers(0, 1 << 32, size=200_000, dtype=np.uint64)
    bits = np.concatenate([bits, rnd.astype(np.uint32)])
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()


def _same_value(a: np.ndarray, b: np.ndarray) -> bool:
    """Equal as numbers, with infinities equal and signed zeros kept apart."""
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_bf16_round_equals_torch_conversion_on_every_pattern_class():
    x = _patterns()
    got = e.bf16_round(x)
    ref = _torch_bf16(x)
    bad = ~(got.view(np.uint32) == ref.view(np.uint32))
    assert not bad.any(), (x[bad][:5], got[bad][:5], ref[bad][:5])


def test_bf16_round_ties_go_to_even_and_overflow_to_infinity():
    # exact ties between two BF16 neighbours
    tie_even = np.array([0x3F808000], dtype=np.uint32).view(np.float32)   # 1 + 2^-8: down to 1
    tie_odd = np.array([0x3F818000], dtype=np.uint32).view(np.float32)    # up to 1 + 2^-6
    assert e.bf16_round(tie_even)[0] == 1.0
    assert e.bf16_round(tie_odd)[0] == np.float32(1.0 + 2.0 ** -6)
    # the largest finite BF16 (0x7F7F) plus half an ulp rounds to +inf
    top = np.array([0x7F7F7FFF, 0x7F7F8000, 0xFF7F8000], dtype=np.uint32).view(np.float32)
    r = e.bf16_round(top)
    assert r[0] == np.array([0x7F7F0000], dtype=np.uint32).view(np.float32)[0]
    assert r[1] == np.inf and r[2] == -np.inf


def _round_half_up(x: np.ndarray) -> np.ndarray:
    """A plausible slip of bf16_round: ties rounded away from zero."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((b + 0x8000) >> 16) << 16).astype(np.uint32).view(np.float32)


def test_the_pin_rejects_a_round_half_up_variant():
    x = _patterns()
    assert not _same_value(_round_half_up(x), _torch_bf16(x))
    assert _same_value(e.bf16_round(x), _torch_bf16(x))


def test_ulp_distance_counts_nextafter_steps():
    g = torch.Generator().manual_seed(9)
    # non-negative BF16 values from the Table 2 range (2^-126 .. 2^8)
    base = torch.exp2(torch.empty(4000).uniform_(-126, 8, generator=g)).to(torch.bfloat16)
    inf = torch.full_like(base, float("inf"))
    cur = base.clone()
    for steps in range(0, 6):
        a = base.float().numpy()
        b = cur.float().numpy()
        assert (e.bf16_ulp_distance(a, b) == steps).all()
        assert (e.bf16_ulp_distance(b, a) == steps).all()
        cur = torch.nextafter(cur, inf)
    # across a power of two the spacing doubles, the count of values does not
    one = torch.tensor([1.0], dtype=torch.bfloat16)
    below = torch.nextafter(one, torch.tensor([0.0], dtype=torch.bfloat16))
    above = torch.nextafter(one, torch.tensor([2.0], dtype=torch.bfloat16))
    assert e.bf16_ulp_distance(below.float().numpy(), above.float().numpy())[0] == 2
