"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test is chosen so a plausible slip in ``oracle/ref_attn.c`` (a dropped
term, a wrong sign or index, a transposed operand, a wrong head mapping or
mask alignment) fails at least one of them. The definition pinned is the
one the FlashAttention-4 method reaches exactly ("FlashAttention-4:
Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
Method and §3.1.4).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attn as oracle
import workloads


def _f64(t):
    return t.to(torch.float64).numpy()


def _dots(q, k, scale):
    """[B,Hq,Sq,Sk] scaled logits via einsum (used for closed forms only)."""
    B, Sq, Hq, d = q.shape
    Hkv = k.shape[2]
    kk = np.repeat(_f64(k), Hq // Hkv, axis=2)
    return scale * np.einsum("bihe,bjhe->bhij", _f64(q), kk)


def test_single_key_gives_that_value_row():
    q, k, v = workloads.make_custom(2, 4, 2, 7, 1, 16, seed=1)
    scale = 0.3
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=False)
    vv = np.repeat(_f64(v), 2, axis=2)            # kv head g serves q heads 2g, 2g+1
    for i in range(7):
        np.testing.assert_allclose(o[:, i], vv[:, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, _dots(q, k, scale)[..., 0], rtol=1e-14, atol=1e-14)


def test_constant_value_rows_give_that_constant():
    q, k, _ = workloads.make_custom(1, 2, 2, 33, 45, 8, seed=2)
    row = torch.linspace(-3, 3, 8).to(torch.bfloat16)
    v = row.view(1, 1, 1, 8).expand(1, 45, 2, 8).contiguous()
    for causal in (False, True):
        o, _ = oracle.attention_fwd(q, k, v, 0.25, causal=causal)
        valid = slice(0, 33) if not causal else slice(0, 33)
        np.testing.assert_allclose(o[:, valid], np.broadcast_to(_f64(row), o[:, valid].shape),
                                   rtol=0, atol=1e-14)


def test_two_keys_reduce_to_a_sigmoid():
    q, k, v = workloads.make_custom(1, 3, 3, 5, 2, 8, seed=3)
    scale = 0.7
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=False)
    x = _dots(q, k, scale)                         # [1,3,5,2]
    sig = 1.0 / (1.0 + np.exp(-(x[..., 1] - x[..., 0])))   # weight of key 1
    vv = _f64(v)
    expect = vv[:, 0][:, None, :, :] + sig.transpose(0, 2, 1)[..., None] * (
        vv[:, 1] - vv[:, 0])[:, None, :, :]
    np.testing.assert_allclose(o, expect, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, np.logaddexp(x[..., 0], x[..., 1]), rtol=1e-14, atol=1e-14)


def test_one_hot_routing_catches_transposed_operands():
    # q_i = 64 e_{pi(i)}, k_j = e_j: row i must pick exactly value row pi(i).
    S, d = 6, 8
    pi = [2, 0, 5, 1, 3, 4]                        # not an involution
    q = torch.zeros(1, S, 1, d)
    k = torch.zeros(1, S, 1, d)
    for i in range(S):
        q[0, i, 0, pi[i]] = 64.0
        k[0, i, 0, i] = 1.0
    v = torch.randn(1, S, 1, d, generator=torch.Generator().manual_seed(4))
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=False)
    for i in range(S):
        np.testing.assert_allclose(o[0, i, 0], _f64(v)[0, pi[i], 0], rtol=0, atol=1e-20)
        assert lse[0, 0, i] == pytest.approx(64.0 + math.log1p((S - 1) * math.exp(-64.0)),
                                             abs=1e-13)


def test_causal_first_row_sees_only_key_zero():
    q, k, v = workloads.make_custom(2, 2, 2, 9, 9, 16, seed=5)
    o, lse = oracle.attention_fwd(q, k, v, 0.25, causal=True)
    np.testing.assert_allclose(o[:, 0], _f64(v)[:, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], _dots(q, k, 0.25)[:, :, 0, 0], rtol=1e-14)


def test_probability_rows_sum_to_one_and_respect_the_mask():
    q, k, v = workloads.make_custom(1, 2, 1, 11, 17, 8, seed=6, dist="wide")
    for causal in (False, True):
        for h in range(2):
            p = oracle.attention_probs(q, k, v, 0.5, causal, b=0, h=h)
            assert (p >= 0).all()
            np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
            if causal:   # bottom-right alignment: key j allowed iff j <= i + (Sk - Sq)
                i, j = np.indices(p.shape)
                assert (p[j > i + (17 - 11)] == 0).all()
                assert (p[j <= i + (17 - 11)] > 0).all()


def test_gqa_equals_repeated_kv_heads():
    q, k, v = workloads.make_custom(2, 8, 2, 13, 21, 16, seed=7)
    rep = lambda t: t.repeat_interleave(4, dim=2).contiguous()  # contiguous head groups
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, 0.25, causal)
        o2, l2 = oracle.attention_fwd(q, rep(k), rep(v), 0.25, causal)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_key_permutation_equivariance():
    q, k, v = workloads.make_custom(1, 2, 2, 10, 19, 8, seed=8)
    perm = torch.randperm(19, generator=torch.Generator().manual_seed(9))
    o1, l1 = oracle.attention_fwd(q, k, v, 0.4, False)
    o2, l2 = oracle.attention_fwd(q, k[:, perm].contiguous(), v[:, perm].contiguous(), 0.4,
                                  False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_dominant_key_selects_its_value_row():
    q, k, v = workloads.make_custom(1, 1, 1, 4, 30, 8, seed=10)
    qf = q.float()
    qf[0, :, 0, :] = 0.0
    qf[0, :, 0, 0] = 1.0
    kf = torch.zeros_like(k, dtype=torch.float32)
    kf[0, 17, 0, 0] = 50.0                         # key 17 wins by +50 nats
    o, _ = oracle.attention_fwd(qf.bfloat16(), kf.bfloat16(), v, 1.0, False)
    for i in range(4):
        np.testing.assert_allclose(o[0, i, 0], _f64(v)[0, 17, 0],
                                   atol=30 * math.exp(-50) * 10)


def test_rows_without_a_valid_key_give_zero_and_minus_inf():
    # Causal with Sq > Sk: rows i < Sq - Sk see no key under bottom-right alignment.
    q, k, v = workloads.make_custom(1, 1, 1, 12, 5, 8, seed=11)
    o, lse = oracle.attention_fwd(q, k, v, 0.3, causal=True)
    assert (o[0, :7] == 0).all() and np.isneginf(lse[0, 0, :7]).all()
    np.testing.assert_allclose(o[0, 7, 0], _f64(v)[0, 0, 0], atol=1e-15)
    assert np.isfinite(lse[0, 0, 7:]).all()


def test_scale_moves_between_q_and_scale():
    q, k, v = workloads.make_custom(1, 2, 2, 9, 14, 16, seed=12)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.5, True)
    o2, l2 = oracle.attention_fwd((q.float() * 2).bfloat16(), k, v, 0.25, True)  # exact in bf16
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_common_key_shift_moves_lse_only():
    g = torch.Generator().manual_seed(13)
    q = torch.randint(-3, 4, (1, 6, 1, 8), generator=g).float()
    k = torch.randint(-3, 4, (1, 10, 1, 8), generator=g).float()
    v = torch.randn(1, 10, 1, 8, generator=g)
    u = torch.randint(-2, 3, (8,), generator=g).float()
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    o1, l1 = oracle.attention_fwd(q, k, v, 0.125, False)
    o2, l2 = oracle.attention_fwd(q, (k.float() + u).bfloat16(), v, 0.125, False)
    shift = 0.125 * (q.double()[0, :, 0, :] @ u.double()).numpy()
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2[0, 0] - l1[0, 0], shift, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", [(2, 4, 2, 37, 37, 16, True), (1, 3, 1, 20, 33, 8, True),
                                   (2, 2, 2, 24, 17, 32, False), (1, 6, 3, 64, 64, 64, True)])
def test_against_torch_sdpa_fp64(shape):
    """Library cross-check: torch's math SDPA in fp64 with an explicit mask."""
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=14)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    qt = q.double().permute(0, 2, 1, 3)
    kt = k.double().repeat_interleave(Hq // Hkv, dim=2).permute(0, 2, 1, 3)
    vt = v.double().repeat_interleave(Hq // Hkv, dim=2).permute(0, 2, 1, 3)
    mask = None
    if causal:
        i = torch.arange(Sq).view(Sq, 1)
        j = torch.arange(Sk).view(1, Sk)
        mask = j <= i + (Sk - Sq)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-11, atol=1e-12)
    logits = scale * qt @ kt.transpose(-1, -2)
    if mask is not None:
        logits = logits.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12,
                               atol=1e-12)


def test_row_subset_matches_full_output():
    w = workloads.Workload("t", 2, 4, 2, 70, 70, 32, True)
    q, k, v = workloads.make_inputs(w, seed=3)
    o, lse = oracle.attention_fwd(q, k, v, w.scale, w.causal)
    rows = workloads.sample_rows(w, n_random=40, seed=1, edge=5)
    o_r, l_r = oracle.attention_fwd_rows(q, k, v, w.scale, w.causal, rows)
    o_g, l_g = oracle.gather_rows(o, lse, rows.numpy(), w.Hq, w.Sq)
    np.testing.assert_array_equal(o_r, o_g)
    np.testing.assert_array_equal(l_r, l_g)


def test_bad_arguments_are_rejected():
    q, k, v = workloads.make_custom(1, 3, 2, 4, 4, 8, seed=0)    # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, 0.5, False)
