"""Pins of the FP8 oracle (oracle/fp8.py): the e4m3 decoder against the
format's defining values and torch's own conversion, the forward against
the C definition (two independent computations), a brute-force tiny case,
and the P-rounding bound against a model of rounding P to e4m3."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn as oracle
from oracle import fp8


# (code, value) from the E4M3 definition: bias 7, 3 mantissa bits, subnormals
# at exponent 0, NaN at S.1111.111, largest finite 448.
DEFINED = [(0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
           (0x30, 0.5), (0x38, 1.0), (0x39, 1.125), (0x3C, 1.5), (0x40, 2.0),
           (0x7E, 448.0), (0x77, 240.0), (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9))]


def test_e4m3_defined_values():
    codes = np.array([c for c, _ in DEFINED], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.e4m3_to_float(codes), [v for _, v in DEFINED])
    assert np.isnan(fp8.e4m3_to_float(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    assert math.copysign(1.0, fp8.e4m3_to_float(np.array([0x80], np.uint8))[0]) == -1.0


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_to_float(codes.numpy())
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (1, 2, 2, 40, 70, 16, False),
    (2, 4, 2, 50, 30, 8, True),      # GQA, Sq > Sk: leading rows see no key
    (1, 2, 1, 33, 90, 32, True),     # Sq < Sk, bottom-right causal
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_fp8_forward_equals_c_definition_on_dequantised_codes(case):
    # e4m3 values are exact in BF16, so the C definition can take the codes
    # as BF16 values with the per-tensor scales folded in:
    #   scale (qs q8)(ks k8)^T = (scale qs ks) q8 k8^T,  softmax(.) (vs v8) = vs softmax(.) v8
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(B, Hq, Hkv, Sq, Sk, d, seed=3)
    o, lse, bound, rss = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, 0.2, causal)

    def as_bf16(t):
        x = torch.from_numpy(fp8.e4m3_to_float(fp8.codes_of(t)))
        xb = x.to(torch.bfloat16)
        assert torch.equal(xb.to(torch.float64), x)
        return xb

    o_c, lse_c = oracle.attention_fwd(as_bf16(q8), as_bf16(k8), as_bf16(v8), 0.2 * qs * ks, causal)
    np.testing.assert_allclose(o, vs * o_c, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_c))
    fin = np.isfinite(lse_c)
    np.testing.assert_allclose(lse[fin], lse_c[fin], rtol=0, atol=1e-12)
    assert (bound >= rss - 1e-15).all() and (bound >= 0).all()


def test_fp8_forward_brute_force_tiny():
    B, Hq, Hkv, Sq, Sk, d = 1, 2, 1, 3, 4, 4
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(B, Hq, Hkv, Sq, Sk, d, seed=9)
    o, lse, _, _ = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, 0.5, True)

    def val(t, s, *idx):
        return float(t[idx].to(torch.float64)) * s

    for h in range(Hq):
        for i in range(Sq):
            keys = [j for j in range(Sk) if j <= i + Sk - Sq]
            sc = [0.5 * sum(val(q8, qs, 0, i, h, e) * val(k8, ks, 0, j, 0, e) for e in range(d))
                  for j in keys]
            z = sum(math.exp(x) for x in sc)
            assert abs(lse[0, h, i] - math.log(z)) < 1e-12
            for e in range(d):
                ref = sum(math.exp(x) / z * val(v8, vs, 0, j, 0, e) for x, j in zip(sc, keys))
                assert abs(o[0, i, h, e] - ref) < 1e-12


@pytest.mark.parametrize("shift", [0.0, 3.0, 8.0])
@pytest.mark.parametrize("dist", ["randn", "wide"])
def test_rounding_bound_covers_e4m3_rounding_of_p(shift, dist):
    # Model of the kernel's rounding: P scaled by 2^shift (a stale row
    # maximum), rounded to e4m3 by torch's conversion, the row sum taken
    # from the unrounded values; the error must stay within `bound`, and the
    # rms ratio to `rss` must be of order one (not vacuous, not exceeded).
    B, Hq, Hkv, Sq, Sk, d = 1, 2, 2, 64, 700, 128
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(B, Hq, Hkv, Sq, Sk, d, seed=4, dist=dist)
    scale = 1.0 / math.sqrt(d)
    o, _, bound, rss = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, scale, False)
    Q = fp8.e4m3_to_float(fp8.codes_of(q8)) * qs
    K = fp8.e4m3_to_float(fp8.codes_of(k8)) * ks
    V = fp8.e4m3_to_float(fp8.codes_of(v8)) * vs
    ratios = []
    for h in range(Hq):
        s = scale * Q[0, :, h, :] @ K[0, :, h, :].T
        p = np.exp(s - s.max(axis=1, keepdims=True)) * 2.0 ** shift
        pr = torch.from_numpy(p).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        o_model = (pr @ V[0, :, h, :]) / p.sum(axis=1, keepdims=True)
        err = np.abs(o_model - o[0, :, h, :])
        assert (err <= bound[0, :, h, :] * (1 + 1e-9)).all()
        ratios.append(np.sqrt(np.mean((err / rss[0, :, h, :]) ** 2)))
    assert 0.05 < max(ratios) < 1.0, ratios


def test_quantised_inputs_use_the_e4m3_range():
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(1, 2, 2, 256, 256, 128, seed=1)
    for t, s in ((q8, qs), (k8, ks), (v8, vs)):
        x = fp8.e4m3_to_float(fp8.codes_of(t))
        assert np.isfinite(x).all() and np.abs(x).max() == 448.0
        assert 0.5 < np.std(x * s) < 2.0
