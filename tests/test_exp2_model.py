"""Pins of the software 2^x model ("FlashAttention-4: Algorithm and Kernel
Pipelining Co-Design for Asymmetric Hardware Scaling", §3.1.3, Table 2)."""
import numpy as np

from oracle import exp2_emu as e
from tests import golden


def test_integers_are_exact_powers_of_two():
    n = np.arange(-126, 9, dtype=np.float32)
    np.testing.assert_array_equal(e.exp2_emulated(n), np.exp2(n.astype(np.float64)))
    assert e.exp2_emulated(np.float32([0.0]))[0] == 1.0


def test_degree3_minimax_error_and_equioscillation():
    (c1, c2, c3), err = e.fit_minimax(3)
    assert err < 2.0 ** -13          # relative error of the polynomial itself
    f = np.linspace(0, 1, 200001)
    rel = (1 + f * (c1 + f * (c2 + f * c3))) / np.exp2(f) - 1
    assert abs(np.abs(rel).max() - err) < 1e-7
    # Chebyshev alternation: >= 4 extrema of alternating sign at +-err.
    ext = np.where(np.abs(np.abs(rel) - err) < 2e-7)[0]
    signs = np.sign(rel[ext])
    runs = 1 + int((np.diff(signs) != 0).sum())
    assert runs >= 4


def test_degree5_reaches_fp32_level():
    _, err5 = e.fit_minimax(5)
    assert err5 < 2.0 ** -22


def test_table2_degree3_within_one_bf16_ulp_on_99_percent():
    # Every BF16 input whose 2^x is a normal fp32 number and that the
    # lazily rescaled softmax can produce (t - m~ <= tau = 8).
    x = e.bf16_grid(-126.0, 8.0)
    got = e.bf16_round(e.exp2_emulated(x))
    ref = e.bf16_round(np.exp2(x.astype(np.float64)).astype(np.float32))
    dist = e.bf16_ulp_distance(got, ref)
    t = golden.load("table2_exp2_bf16.txt")       # the pages' claim, with its citation
    assert (dist <= t["max_bf16_ulp"]).mean() >= t["min_fraction_within"]
    assert dist.max() <= 1


def test_monotone_on_the_bf16_grid():
    x = e.bf16_grid(-126.0, 8.0)
    y = e.bf16_round(e.exp2_emulated(x))
    assert (np.diff(y.astype(np.float64)) >= 0).all()


def test_below_the_normal_range_the_result_is_negligible():
    x = np.float32([-126.5, -127.0, -300.0, -np.inf])
    y = e.exp2_emulated(x)
    assert (y >= 0).all() and (y < 2.0 ** -126).all()
