"""GPU parity of the CUDA forward pass against the fp64 oracle.

Every call goes through the C ABI (``attention_forward_fa4_gb300`` is a
ctypes binding). Small shapes are compared element by element on every
output; the full-size workloads are compared on a deterministic row
sample (first and last rows of each head plus seeded random rows) in the
same launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn as oracle
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


def _run(q, k, v, causal, scale=None, **kw):
    fa4 = _fa4()
    o, lse = fa4.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, **kw)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    return o, lse


def _full_check(q, k, v, causal, scale, what, **kw):
    o, lse = _run(q, k, v, causal, scale, **kw)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, scale, causal)
    return parity.assert_close(parity.to_np(o), parity.to_np(lse), o_ref, lse_ref, what)


# ------------------------------------------------------------ small, every element
EDGE_CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (1, 2, 2, 256, 256, 64, False),     # the tiny workload shape
    (1, 2, 2, 256, 256, 64, True),
    (2, 4, 4, 200, 200, 128, False),    # ragged tail in both tiles
    (2, 4, 4, 200, 200, 128, True),
    (1, 8, 2, 300, 300, 128, True),     # GQA 4:1, three query tiles
    (1, 2, 2, 130, 700, 64, True),      # Sq < Sk, bottom-right causal
    (1, 2, 2, 700, 130, 128, True),     # Sq > Sk: leading rows see no key
    (1, 2, 1, 1, 1, 128, False),        # single query, single key
    (1, 3, 3, 64, 5, 64, False),        # fewer keys than one block, tile 1 empty
    (3, 2, 2, 129, 257, 64, False),     # one row into tile 1, one key into block 2
    (1, 1, 1, 512, 512, 128, True),     # two full CTAs, diagonal blocks
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("emu", [0, 8, 4], ids=["mufu", "emu8", "emu4"])
def test_small_shapes_match_oracle(case, emu):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=31)
    _full_check(q, k, v, causal, 1.0 / math.sqrt(d), str(case), exp2_emulation=emu)


@pytest.mark.parametrize("cwg", [False, True], ids=["inline", "corr_wg"])
def test_large_logits_match_oracle(cwg):
    # |scores| ~ 16 x larger: row maxima jump between blocks, rescales fire.
    q, k, v = workloads.make_custom(2, 2, 2, 384, 640, 128, seed=32, dist="wide")
    for causal in (False, True):
        _full_check(q, k, v, causal, 1 / math.sqrt(128), f"wide causal={causal}",
                    correction_warpgroup=cwg)


@pytest.mark.parametrize("cwg", [False, True], ids=["inline", "corr_wg"])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_eager_and_lazy_rescale_both_match(tau, cwg):
    w = workloads.Workload("ramp", 1, 4, 1, 1024, 1024, 128, True, ramp=0.03)
    q, k, v = workloads.make_inputs(w, seed=0)
    _full_check(q, k, v, True, w.scale, f"tau={tau}", tau=tau, correction_warpgroup=cwg)


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: "x".join(map(str, c)))
def test_small_shapes_with_correction_warpgroup(case):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=31, dist="wide")
    _full_check(q, k, v, causal, 1.0 / math.sqrt(d), str(case), correction_warpgroup=True)


@pytest.mark.parametrize("shape", [(2, 4, 4, 1100, 1300, 128, True), (1, 8, 2, 900, 2100, 64, False),
                                   (2, 4, 2, 700, 700, 64, True)])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_correction_modes_agree_bit_for_bit(shape, tau):
    """The softmax warp rescaling its own rows and the correction warpgroup
    doing it compute the same products in the same order."""
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=44, dist="wide")
    o1, l1 = _run(q, k, v, causal, tau=tau, correction_warpgroup=False)
    o2, l2 = _run(q, k, v, causal, tau=tau, correction_warpgroup=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lazy_and_eager_agree_to_bf16_noise():
    w = workloads.Workload("ramp", 1, 4, 1, 1024, 1024, 128, True, ramp=0.03)
    q, k, v = workloads.make_inputs(w, seed=0)
    o8, l8 = _run(q, k, v, True, w.scale, tau=8.0)
    o0, l0 = _run(q, k, v, True, w.scale, tau=0.0)
    assert (o8.float() - o0.float()).abs().max().item() <= 2e-2
    assert (l8 - l0).abs().max().item() <= 1e-4


def test_no_keys_and_no_queries():
    fa4 = _fa4()
    q, k, v = workloads.make_custom(1, 2, 2, 40, 1, 64, seed=33)
    qd = q.to(DEV)
    kd = torch.empty((1, 0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o, lse = fa4.fwd(qd, kd, kd.clone(), causal=False)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    qe = torch.empty((1, 0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o, lse = fa4.fwd(qe, k.to(DEV), v.to(DEV), causal=True)
    assert o.numel() == 0 and lse.numel() == 0


def test_gqa_equals_repeated_heads_on_gpu():
    q, k, v = workloads.make_custom(1, 8, 2, 256, 384, 128, seed=34)
    rep = lambda t: t.repeat_interleave(4, dim=2).contiguous()
    o1, l1 = _run(q, k, v, True)
    o2, l2 = _run(q, rep(k), rep(v), True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_constant_values_and_single_key_on_gpu():
    q, k, _ = workloads.make_custom(1, 2, 2, 300, 300, 128, seed=35)
    row = torch.linspace(-2, 2, 128).to(torch.bfloat16)
    v = row.view(1, 1, 1, 128).expand(1, 300, 2, 128).contiguous()
    o, _ = _run(q, k, v, True)
    assert (o.float().cpu() - row.float()).abs().max().item() <= 2e-2
    q1, k1, v1 = workloads.make_custom(2, 4, 2, 50, 1, 64, seed=36)
    o, lse = _run(q1, k1, v1, False, 0.125)
    vv = v1.repeat_interleave(2, dim=2).float()
    assert (o.float().cpu() - vv[:, 0:1].expand(2, 50, 4, 64)).abs().max().item() <= 2e-2


def test_rescale_counter_lazy_below_eager():
    w = workloads.Workload("ramp", 1, 8, 2, 2048, 2048, 128, True, ramp=0.02)
    q, k, v = workloads.make_inputs(w, seed=0)
    counts = {}
    for tau in (0.0, 8.0):
        stats = torch.zeros(2, dtype=torch.int64, device=DEV)
        _run(q, k, v, True, w.scale, tau=tau, rescale_stats=stats)
        counts[tau] = stats.cpu().tolist()
    assert counts[0.0][1] == counts[8.0][1] > 0
    assert counts[8.0][0] < counts[0.0][0]


# ------------------------------------------------------------ full-size workloads
FULL = [workloads.TINY, workloads.MID, workloads.LONG_CAUSAL, workloads.GQA_STRESS] + \
    workloads.d64_sweep()


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_workload_matches_oracle_on_sampled_rows(w):
    q, k, v = workloads.make_inputs(w, seed=0)
    o, lse = _run(q, k, v, w.causal, w.scale)
    if w is workloads.TINY:
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, w.causal)
        parity.assert_close(parity.to_np(o), parity.to_np(lse), o_ref, lse_ref, w.name)
        return
    n_bh = w.B * w.Hq
    rows = workloads.sample_rows(w, n_random=512, seed=1, edge=32, max_bh=min(n_bh, 8))
    o_ref, lse_ref = oracle.attention_fwd_rows(q, k, v, w.scale, w.causal, rows)
    o_g, l_g = parity.gather_gpu_rows(o, lse, rows)
    parity.assert_close(o_g, l_g, o_ref, lse_ref, w.name)
    # properties that hold at any size: finite outputs everywhere
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# ------------------------------------------------------------ 2^x emulation
def test_exp2_emulation_table2_on_device():
    """Every finite BF16 input with a normal result: the degree-3 emulation,
    rounded to BF16, is within 1 BF16 ULP of exact 2^x on >= 99 % of them
    ("FlashAttention-4", §3.1.3, Table 2), and also vs MUFU.EX2."""
    fa4 = _fa4()
    bits = (torch.arange(0, 1 << 16, dtype=torch.int32) << 16)
    x = bits.view(torch.float32)
    x = x[torch.isfinite(x) & (x >= -126.0) & (x <= 8.0)].contiguous()
    ye, ym = fa4.exp2_eval(x.to(DEV))
    torch.cuda.synchronize()
    ye = ye.cpu().numpy()
    ym = ym.cpu().numpy()
    from oracle import exp2_emu as e
    exact = np.exp2(x.numpy().astype(np.float64)).astype(np.float32)
    d_exact = e.bf16_ulp_distance(e.bf16_round(ye), e.bf16_round(exact))
    d_mufu = e.bf16_ulp_distance(e.bf16_round(ye), e.bf16_round(ym))
    assert (d_exact <= 1).mean() >= 0.99, (d_exact <= 1).mean()
    assert (d_mufu <= 1).mean() >= 0.99, (d_mufu <= 1).mean()
    ints = torch.arange(-126, 9, dtype=torch.float32)
    yi, _ = fa4.exp2_eval(ints.to(DEV))
    assert torch.equal(yi.cpu(), torch.exp2(ints))


# ------------------------------------------------------------ MMA issue order
@pytest.mark.parametrize("shape", [(2, 16, 16, 2048, 2048, 128, True),
                                   (1, 8, 2, 1536, 1536, 128, False),
                                   (4, 8, 8, 1024, 1024, 64, True)])
def test_back_to_back_issue_equals_strict_order(shape):
    """The next S MMA is issued right behind the P*V MMA that reads the same
    tensor-memory columns; waiting for the P*V first must give bit-identical
    output (repeated, to catch a rare reordering)."""
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=41, dist="wide")
    o_s, l_s = _run(q, k, v, causal, strict_mma_order=True)
    for _ in range(5):
        o_f, l_f = _run(q, k, v, causal)
        assert torch.equal(o_f, o_s) and torch.equal(l_f, l_s)


# ------------------------------------------------------------ grid modes
@pytest.mark.parametrize("shape", [(2, 8, 8, 2048, 2048, 128, True),
                                   (3, 4, 2, 700, 900, 64, False),
                                   (1, 8, 8, 1536, 1536, 64, True)])
def test_grid_modes_agree_bit_for_bit(shape):
    """One CTA per work tile and the persistent grid (snake order) compute
    identical outputs."""
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=43)
    o1, l1 = _run(q, k, v, causal, grid_mode=1)
    o2, l2 = _run(q, k, v, causal, grid_mode=2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------ own P columns
# At head dim 64 the persistent grid keeps P_t in its own tensor-memory
# columns and computes S_t(j+1) while softmax_t(j) runs. The shapes give
# more work tiles than SMs, so CTAs run several tiles back to back (the
# hand-offs of S, P and O across tiles), with ragged tails, GQA and wide
# logits (frequent rescales).
OWN_P_SHAPES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (2, 40, 8, 300, 700, 64, True),
    (2, 40, 8, 300, 700, 64, False),
    (1, 80, 80, 520, 260, 64, True),
]


@pytest.mark.parametrize("cwg", [False, True], ids=["inline", "corr_wg"])
@pytest.mark.parametrize("shape", OWN_P_SHAPES, ids=lambda c: "x".join(map(str, c)))
def test_own_p_persistent_matches_oracle(shape, cwg):
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=45, dist="wide")
    _full_check(q, k, v, causal, 1.0 / math.sqrt(d), f"own P {shape}", grid_mode=2,
                correction_warpgroup=cwg)


@pytest.mark.parametrize("tau", [0.0, 8.0])
@pytest.mark.parametrize("shape", [(4, 32, 8, 1024, 1024, 64, True), (8, 16, 16, 777, 1200, 64, False)],
                         ids=lambda c: "x".join(map(str, c)))
def test_own_p_equals_aliased_p_bit_for_bit(shape, tau):
    """The persistent grid (own P columns, several tiles per CTA) and one CTA
    per work tile (P aliasing S) compute the same products in the same
    order: identical outputs, in both correction modes."""
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=46, dist="wide")
    o1, l1 = _run(q, k, v, causal, tau=tau, grid_mode=1)
    for cwg in (False, True):
        o2, l2 = _run(q, k, v, causal, tau=tau, grid_mode=2, correction_warpgroup=cwg)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
