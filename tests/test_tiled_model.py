"""The conditional rescale is exact algebra: the fp64 tiled model equals the
definition for every threshold tau ("FlashAttention-4: Algorithm and Kernel
Pipelining Co-Design for Asymmetric Hardware Scaling", §3.1.4, Eq. 6: the
final 1/l normalisation recovers the exact result)."""
import numpy as np
import pytest
import torch

from oracle import attn as oracle
from oracle import tiled_model
import workloads

CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal, dist
    (1, 2, 2, 256, 256, 64, False, "randn"),
    (1, 2, 1, 200, 200, 32, True, "wide"),     # ragged tail, GQA, causal
    (2, 2, 2, 130, 300, 16, True, "wide"),     # Sq != Sk, bottom-right mask
    (1, 1, 1, 64, 40, 16, True, "randn"),      # Sq > Sk: rows with no key
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("tau", [0.0, 8.0, 1e9])
def test_tiled_model_equals_definition(case, tau):
    B, Hq, Hkv, Sq, Sk, d, causal, dist = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=21, dist=dist)
    scale = d ** -0.5
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, scale, causal)
    o, lse, _ = tiled_model.tiled_attention_fwd(q, k, v, scale, causal, tau=tau)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lse_ref)
    assert (np.isfinite(lse) == fin).all()
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)


def test_lazy_rescale_skips_rescales_on_a_rising_max():
    # Rising keys (the GQA stress recipe, shrunk): row maxima keep climbing.
    w = workloads.Workload("ramp", 1, 4, 1, 1024, 1024, 64, True, ramp=0.03)
    q, k, v = workloads.make_inputs(w, seed=0)
    _, _, eager = tiled_model.tiled_attention_fwd(q, k, v, w.scale, True, tau=0.0)
    _, _, lazy = tiled_model.tiled_attention_fwd(q, k, v, w.scale, True, tau=8.0)
    assert eager["group_blocks"] == lazy["group_blocks"] > 0
    assert lazy["rescaled_group_blocks"] < eager["rescaled_group_blocks"]


def test_probabilities_stay_below_two_to_the_tau():
    # With the reference max lagging by at most tau, no p exceeds 2^tau.
    q, k, v = workloads.make_custom(1, 1, 1, 128, 512, 32, seed=5, dist="wide")
    scale = 32 ** -0.5
    c = scale / np.log(2.0)
    qf, kf = q.double().numpy()[0, :, 0], k.double().numpy()[0, :, 0]
    t = c * qf @ kf.T
    m_ref = np.full(128, -np.inf)
    worst = 0.0
    for j0 in range(0, 512, 128):
        blk = t[:, j0:j0 + 128]
        m_new = np.maximum(m_ref, blk.max(1))
        need = m_new > m_ref + 8.0
        gate = np.repeat(need.reshape(4, 32).any(1), 32)
        m_ref = np.where(gate, m_new, m_ref)
        worst = max(worst, float(np.exp2(blk - m_ref[:, None]).max()))
    assert worst <= 256.0
