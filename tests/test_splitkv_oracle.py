"""Pins of the key-range split model (oracle/splitkv.py): the key-range
forward against the C definition, and the combine against the unsplit
definition -- two independent computations."""
import numpy as np
import pytest

import workloads
from oracle import attn as oracle
from oracle import splitkv as sk

CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (1, 2, 2, 37, 300, 16, False),
    (2, 4, 2, 50, 260, 8, True),       # GQA, Sq < Sk (bottom-right causal)
    (1, 2, 1, 90, 40, 8, True),        # Sq > Sk: leading rows see no key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_full_key_range_equals_the_definition(case):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=5)
    o, lse = sk.keyrange_fwd(q, k, v, 0.3, causal, 0, Sk)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("cuts", [(0, 1), (0, 100, 101, 200), (0, 7, 129, 130, 256)])
def test_merge_of_a_partition_equals_the_definition(case, cuts):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=6)
    edges = sorted(set([c for c in cuts if c < Sk] + [Sk]))
    parts = [sk.keyrange_fwd(q, k, v, 0.3, causal, a, b) for a, b in zip(edges[:-1], edges[1:])]
    o, lse = sk.merge([p[0] for p in parts], [p[1] for p in parts])
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isneginf(lse), ~fin)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


def test_empty_range_is_neutral_and_merge_is_order_free():
    q, k, v = workloads.make_custom(1, 2, 2, 40, 200, 8, seed=7)
    # causal with Sq = 40 < Sk = 200: key 199 is visible to the last row only;
    # keys past Sk give an empty range.
    o_e, lse_e = sk.keyrange_fwd(q, k, v, 0.5, True, 200, 260)
    assert (o_e == 0).all() and np.isneginf(lse_e).all()
    a = sk.keyrange_fwd(q, k, v, 0.5, True, 0, 90)
    b = sk.keyrange_fwd(q, k, v, 0.5, True, 90, 200)
    o1, l1 = sk.merge([a[0], b[0], o_e], [a[1], b[1], lse_e])
    o2, l2 = sk.merge([b[0], a[0]], [b[1], a[1]])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)
    o3, l3 = sk.merge([a[0]], [a[1]])                     # a single part is returned unchanged
    np.testing.assert_array_equal(o3, a[0])
    np.testing.assert_allclose(l3, a[1], rtol=0, atol=1e-15)


def test_split_ranges_cover_whole_blocks():
    assert sk.split_ranges(1000, 3) == [(0, 384), (384, 768), (768, 1000)]
    assert sk.split_ranges(300, 8) == [(0, 128), (128, 256), (256, 300)]
    assert sk.split_ranges(128, 1) == [(0, 128)]
    r = sk.split_ranges(20000, 16)
    assert r[0][0] == 0 and r[-1][1] == 20000
    assert all(a1 == b0 for (_, a1), (b0, _) in zip(r[:-1], r[1:]))
