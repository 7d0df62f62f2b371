"""GPU parity of the FP8 (e4m3) forward against the fp64 oracle of the
dequantised inputs (oracle/fp8.py).

Every call goes through the C ABI (``fa4_fwd_fp8``). The tolerance is the
one derived in tests/parity.py (``assert_close_fp8``): an element-wise
worst case from the e4m3 rounding of P and the BF16 rounding of O, a
root-mean-square check against the error scale of that rounding, and the
BF16 path's LSE bound.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import fp8 as oracle8
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


def _run(q8, k8, v8, qs, ks, vs, causal, scale=None, **kw):
    fa4 = _fa4()
    o, lse = fa4.fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), qs, ks, vs, causal=causal,
                         scale=scale, **kw)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    return o, lse


def _full_check(inputs, causal, scale, what, **kw):
    q8, k8, v8, qs, ks, vs = inputs
    o, lse = _run(q8, k8, v8, qs, ks, vs, causal, scale, **kw)
    o_ref, lse_ref, bound, rss = oracle8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, scale, causal)
    return parity.assert_close_fp8(parity.to_np(o), parity.to_np(lse), o_ref, lse_ref, bound,
                                   rss, what)


EDGE_CASES = [
    # B, Hq, Hkv, Sq, Sk, causal (d = 128)
    (2, 4, 4, 200, 200, False),     # ragged tail in both tiles
    (2, 4, 4, 200, 200, True),
    (1, 8, 2, 300, 300, True),      # GQA 4:1, three query tiles
    (1, 2, 2, 130, 700, True),      # Sq < Sk, bottom-right causal
    (1, 2, 2, 700, 130, True),      # Sq > Sk: leading rows see no key
    (1, 2, 1, 1, 1, False),         # single query, single key
    (1, 3, 3, 64, 5, False),        # fewer keys than one block, tile 1 empty
    (3, 2, 2, 129, 257, False),     # one row into tile 1, one key into block 2
    (1, 1, 1, 512, 512, True),      # two full CTAs, diagonal blocks
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("grid_mode", [1, 2], ids=["per_tile", "persistent"])
def test_small_shapes_match_oracle(case, grid_mode):
    B, Hq, Hkv, Sq, Sk, causal = case
    inputs = workloads.make_custom_fp8(B, Hq, Hkv, Sq, Sk, 128, seed=51)
    _full_check(inputs, causal, 1.0 / math.sqrt(128), str(case), grid_mode=grid_mode)


@pytest.mark.parametrize("cwg", [False, True], ids=["inline", "corr_wg"])
def test_large_logits_match_oracle(cwg):
    # |scores| ~ 16 x larger: row maxima jump between blocks, rescales fire.
    inputs = workloads.make_custom_fp8(2, 2, 2, 384, 640, 128, seed=52, dist="wide")
    for causal in (False, True):
        _full_check(inputs, causal, 1 / math.sqrt(128), f"wide causal={causal}",
                    correction_warpgroup=cwg)


@pytest.mark.parametrize("cwg", [False, True], ids=["inline", "corr_wg"])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_eager_and_lazy_rescale_both_match(tau, cwg):
    w = workloads.Workload("ramp", 1, 4, 1, 1024, 1024, 128, True, ramp=0.03)
    inputs = workloads.make_inputs_fp8(w, seed=0)
    _full_check(inputs, True, w.scale, f"tau={tau}", tau=tau, correction_warpgroup=cwg)


def test_scales_enter_as_the_definition_says():
    # Doubling q_scale doubles the logits; doubling v_scale doubles O exactly
    # (a power of two), LSE unchanged.
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(1, 4, 2, 256, 384, 128, seed=53)
    o1, l1 = _run(q8, k8, v8, qs, ks, vs, True)
    o2, l2 = _run(q8, k8, v8, qs, ks, 2.0 * vs, True)
    assert torch.equal(o2.float(), 2.0 * o1.float()) and torch.equal(l1, l2)
    _full_check((q8, k8, v8, 2.0 * qs, ks, 0.75 * vs), True, 0.05, "scaled logits")


def test_gqa_equals_repeated_heads_and_is_deterministic():
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(1, 8, 2, 256, 384, 128, seed=54)
    rep = lambda t: t.view(torch.uint8).repeat_interleave(4, dim=2).contiguous().view(t.dtype)
    o1, l1 = _run(q8, k8, v8, qs, ks, vs, True)
    o2, l2 = _run(q8, rep(k8), rep(v8), qs, ks, vs, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = _run(q8, k8, v8, qs, ks, vs, True)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_back_to_back_issue_equals_strict_order():
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(2, 16, 16, 2048, 2048, 128, seed=55,
                                                       dist="wide")
    o_s, l_s = _run(q8, k8, v8, qs, ks, vs, True, strict_mma_order=True)
    for _ in range(3):
        o_f, l_f = _run(q8, k8, v8, qs, ks, vs, True)
        assert torch.equal(o_f, o_s) and torch.equal(l_f, l_s)


def test_constant_values_give_that_row():
    # V rows all equal to one e4m3 row: the oracle's O is that row times
    # v_scale whatever P is; the kernel's differs only by the e4m3 rounding
    # of P (its row sum adds the unrounded P).
    q8, k8, _, qs, ks, _ = workloads.make_custom_fp8(1, 2, 2, 300, 300, 128, seed=56)
    row = torch.linspace(-2, 2, 128).to(torch.float8_e4m3fn)
    v8 = row.view(1, 1, 1, 128).expand(1, 300, 2, 128).contiguous()
    o_ref, _, _, _ = oracle8.attention_fwd_fp8(q8, k8, v8, qs, ks, 0.5, 1 / math.sqrt(128), True)
    np.testing.assert_allclose(o_ref, np.broadcast_to(0.5 * row.double().numpy(), o_ref.shape),
                               rtol=0, atol=1e-12)
    _full_check((q8, k8, v8, qs, ks, 0.5), True, 1 / math.sqrt(128), "constant V")


def test_no_keys_no_queries_and_rejected_arguments():
    fa4 = _fa4()
    q8, k8, v8, qs, ks, vs = workloads.make_custom_fp8(1, 2, 2, 40, 1, 128, seed=57)
    kd = torch.empty((1, 0, 2, 128), dtype=torch.float8_e4m3fn, device=DEV)
    o, lse = fa4.fwd_fp8(q8.to(DEV), kd, kd.clone(), qs, ks, vs)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    qe = torch.empty((1, 0, 2, 128), dtype=torch.float8_e4m3fn, device=DEV)
    o, lse = fa4.fwd_fp8(qe, k8.to(DEV), v8.to(DEV), qs, ks, vs, causal=True)
    assert o.numel() == 0 and lse.numel() == 0
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), 0.0, ks, vs)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), qs, ks, float("nan"))
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
    q64 = torch.zeros((1, 8, 2, 64), dtype=torch.float8_e4m3fn, device=DEV)
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_fp8(q64, q64.clone(), q64.clone(), 1.0, 1.0, 1.0)
    assert e.value.code == fa4.FA4_ERR_UNSUPPORTED


# ------------------------------------------------------------ full-size workloads
FULL = [workloads.MID, workloads.LONG_CAUSAL, workloads.GQA_STRESS]


@pytest.mark.parametrize("w", FULL, ids=lambda w: "fp8_" + w.name)
def test_workload_matches_oracle_on_sampled_rows(w):
    q8, k8, v8, qs, ks, vs = workloads.make_inputs_fp8(w, seed=0)
    o, lse = _run(q8, k8, v8, qs, ks, vs, w.causal, w.scale)
    n_bh = w.B * w.Hq
    rows = workloads.sample_rows(w, n_random=256, seed=1, edge=32, max_bh=min(n_bh, 4))
    o_ref, lse_ref, bound, rss = oracle8.attention_fwd_fp8_rows(q8, k8, v8, qs, ks, vs, w.scale,
                                                               w.causal, rows.numpy())
    o_g, l_g = parity.gather_gpu_rows(o, lse, rows)
    parity.assert_close_fp8(o_g, l_g, o_ref, lse_ref, bound, rss, w.name)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
