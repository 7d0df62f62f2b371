"""Pins of the fp64 backward reference (oracle/attn_bwd.py) against things
it does not compute itself: central finite differences of an independent
fp64 forward, torch autograd in fp64, the C forward reference, and
closed-form invariants."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attn as oracle
from oracle import attn_bwd as ob


def _fwd_np(q, k, v, scale, causal):
    """Independent plain fp64 forward (for finite differences only)."""
    B, Sq, Hq, d = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    grp = Hq // Hkv
    o = np.zeros((B, Sq, Hq, d))
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                js = [j for j in range(Sk) if not causal or j <= i + Sk - Sq]
                if not js:
                    continue
                x = np.array([scale * q[b, i, h] @ k[b, j, h // grp] for j in js])
                w = np.exp(x - x.max())
                o[b, i, h] = (w[:, None] * v[b, js, h // grp]).sum(0) / w.sum()
    return o


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    B, Hq, Hkv, Sq, Sk, d = 1, 2, 1, 3, 4, 2
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=81)
    g = torch.Generator().manual_seed(82)
    do = torch.randn((B, Sq, Hq, d), generator=g).to(torch.bfloat16)
    scale = 0.7
    ref = ob.attention_bwd(q, k, v, do, scale, causal)
    qf, kf, vf, dof = (t.to(torch.float64).numpy() for t in (q, k, v, do))
    loss = lambda qq, kk, vv: float((_fwd_np(qq, kk, vv, scale, causal) * dof).sum())
    eps = 1e-6
    for name, arr in (("dq", qf), ("dk", kf), ("dv", vf)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args_p = {"dq": (plus, kf, vf), "dk": (qf, plus, vf), "dv": (qf, kf, plus)}[name]
            args_m = {"dq": (minus, kf, vf), "dk": (qf, minus, vf), "dv": (qf, kf, minus)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(ref[name], num, rtol=0, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("shape", [(2, 4, 2, 33, 47, 16, False), (1, 2, 2, 40, 29, 8, True),
                                   (1, 3, 1, 20, 64, 8, True)])
def test_against_torch_autograd_fp64(shape):
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=83)
    do = torch.randn((B, Sq, Hq, d), generator=torch.Generator().manual_seed(84)).to(torch.bfloat16)
    scale = d ** -0.5
    ref = ob.attention_bwd(q, k, v, do, scale, causal)
    grp = Hq // Hkv
    qt = q.to(torch.float64).permute(0, 2, 1, 3).requires_grad_(True)             # [B,Hq,Sq,d]
    kt = k.to(torch.float64).permute(0, 2, 1, 3).requires_grad_(True)
    vt = v.to(torch.float64).permute(0, 2, 1, 3).requires_grad_(True)
    logits = scale * qt @ kt.repeat_interleave(grp, dim=1).transpose(-1, -2)
    if causal:
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        logits = logits.masked_fill(j > i + (Sk - Sq), float("-inf"))
    p = torch.softmax(logits, dim=-1).nan_to_num(0.0)
    o = p @ vt.repeat_interleave(grp, dim=1)
    (o * do.to(torch.float64).permute(0, 2, 1, 3)).sum().backward()
    np.testing.assert_allclose(ref["dq"], qt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ref["dk"], kt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ref["dv"], vt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_forward_part_matches_the_c_definition():
    q, k, v = workloads.make_custom(2, 4, 2, 50, 70, 16, seed=85)
    do = torch.zeros((2, 50, 4, 16), dtype=torch.bfloat16)
    ref = ob.attention_bwd(q, k, v, do, 0.25, True)
    o, lse = oracle.attention_fwd(q, k, v, 0.25, True)
    np.testing.assert_allclose(ref["o"], o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ref["lse"], lse, rtol=0, atol=1e-12)


def test_invariants():
    q, k, v = workloads.make_custom(1, 2, 2, 24, 40, 8, seed=86)
    do = torch.randn((1, 24, 2, 8), generator=torch.Generator().manual_seed(87)).to(torch.bfloat16)
    ref = ob.attention_bwd(q, k, v, do, 0.4, False)
    # rows of P sum to 1, so the value gradients sum (over keys) to the output gradients
    np.testing.assert_allclose(ref["dv"].sum(axis=1), do.double().numpy().sum(axis=1), atol=1e-12)
    # constant V rows: dP rows are constant, dS = 0, so dQ = dK = 0
    vc = torch.ones_like(v) * 0.5
    r2 = ob.attention_bwd(q, k, vc, do, 0.4, False)
    assert np.abs(r2["dq"]).max() < 1e-12 and np.abs(r2["dk"]).max() < 1e-12
    # GQA: the grads of a shared kv head equal the sum over repeated heads
    q4, k1, v1 = workloads.make_custom(1, 4, 1, 16, 20, 8, seed=88)
    do4 = torch.randn((1, 16, 4, 8), generator=torch.Generator().manual_seed(89)).to(torch.bfloat16)
    a = ob.attention_bwd(q4, k1, v1, do4, 0.3, True)
    b = ob.attention_bwd(q4, k1.repeat_interleave(4, dim=2), v1.repeat_interleave(4, dim=2), do4, 0.3,
                         True)
    np.testing.assert_allclose(a["dq"], b["dq"], atol=1e-13)
    np.testing.assert_allclose(a["dk"][:, :, 0], b["dk"].sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(a["dv"][:, :, 0], b["dv"].sum(axis=2), atol=1e-13)
