"""GPU parity of the attention backward (fa4_bwd, through the C ABI)
against the fp64 gradient by the definition (oracle/attn_bwd.py).

Tolerance (per gradient tensor G with reference R): max|G - R| <= 2e-2 +
2e-2 max|R| and mean|G - R| <= 2e-3 + 2e-3 mean|R|. The kernel rounds P and
dS to BF16 before the MMAs and writes BF16 gradients (2^-9 relative each);
the accumulations are fp32."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_bwd as ob

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


def _check(name, got, ref, log):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    mx, mean = err.max() if err.size else 0.0, err.mean() if err.size else 0.0
    ref_mx = np.abs(ref).max() if ref.size else 0.0
    ref_mean = np.abs(ref).mean() if ref.size else 0.0
    log.append(f"{name}: max {mx:.3e} (ref max {ref_mx:.3e}) mean {mean:.3e} (ref mean {ref_mean:.3e})")
    assert mx <= 2e-2 + 2e-2 * ref_mx, log
    assert mean <= 2e-3 + 2e-3 * ref_mean, log


def _bwd_case(B, Hq, Hkv, Sq, Sk, d, causal, seed):
    fa4 = _fa4()
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    do = torch.randn((B, Sq, Hq, d), generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa4.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa4.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    ref = ob.attention_bwd(q, k, v, do, scale, causal)
    log = [str((B, Hq, Hkv, Sq, Sk, d, causal))]
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(name, got, ref[name], log)
    return log


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (1, 2, 2, 256, 256, 64, False),
    (1, 2, 2, 256, 256, 128, True),
    (2, 4, 2, 200, 300, 128, True),     # GQA, ragged, Sq < Sk
    (1, 2, 2, 130, 700, 64, True),      # bottom-right causal
    (1, 2, 2, 700, 130, 128, True),     # Sq > Sk: leading rows see no key
    (1, 1, 1, 1, 1, 128, False),        # single query, single key
    (1, 3, 3, 64, 5, 64, False),        # fewer keys than a block
    (1, 4, 2, 1024, 1024, 128, True),   # several blocks each way
    (1, 2, 1, 320, 320, 128, True),     # GQA; key blocks with 2 and 4 query steps of 64
    (2, 4, 4, 190, 333, 128, False),    # ragged both ways, 3 query steps of 64
    (1, 2, 2, 64, 256, 128, True),      # one 64-query step per head
    (1, 8, 1, 96, 128, 128, False),     # group of 8: 16 steps through one key block
    (2, 4, 2, 200, 300, 64, True),      # head dim 64: GQA, ragged, bottom-right causal
    (1, 8, 1, 96, 128, 64, False),      # head dim 64: 16 steps through one key block
    (1, 2, 2, 1024, 1024, 64, True),    # head dim 64: several blocks each way
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_bwd_matches_oracle(case):
    _bwd_case(*case, seed=91)


def test_bwd_empty_edges():
    fa4 = _fa4()
    q, k, v = (t.to(DEV) for t in workloads.make_custom(1, 2, 2, 40, 64, 64, seed=92))
    # no queries: dk = dv = 0
    qe = torch.empty((1, 0, 2, 64), dtype=torch.bfloat16, device=DEV)
    lse_e = torch.empty((1, 2, 0), dtype=torch.float32, device=DEV)
    dq, dk, dv = fa4.bwd(qe, k, v, qe.clone(), qe.clone(), lse_e)
    torch.cuda.synchronize()
    assert (dk == 0).all() and (dv == 0).all()
    # no keys: dq = 0
    ke = torch.empty((1, 0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros_like(q)
    lse = torch.full((1, 2, 40), float("-inf"), device=DEV)
    dq, dk, dv = fa4.bwd(q, ke, ke.clone(), o, torch.ones_like(q), lse)
    torch.cuda.synchronize()
    assert (dq == 0).all()


@pytest.mark.parametrize("case", [(1, 4, 2, 1024, 2048, 128, True), (2, 2, 2, 700, 900, 64, False)],
                         ids=lambda c: "x".join(map(str, c)))
def test_deterministic_mode_repeats_bit_for_bit_and_matches_oracle(case):
    """fa4_bwd_ex(deterministic=1) adds the key blocks' dQ tiles in key-block
    order: repeated runs agree bit for bit, and the result is the gradient."""
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=93)
    do = torch.randn((B, Sq, Hq, d), generator=torch.Generator().manual_seed(94)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa4.fwd(qd, kd, vd, causal=causal, scale=scale)
    runs = [fa4.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale, deterministic=True)
            for _ in range(3)]
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)
    ref = ob.attention_bwd(q, k, v, do, scale, causal)
    log = [str(case)]
    for name, got in zip(("dq", "dk", "dv"), runs[0]):
        _check(name, got, ref[name], log)


@pytest.mark.parametrize("w", [workloads.MID, workloads.LONG_CAUSAL,
                               workloads.by_name("d64_causal_b8_h32_s4096")], ids=lambda w: w.name)
def test_bwd_full_size_sampled_heads(w):
    """The backward of a full-size workload in the launch the benchmark times
    (its seeded dO included); the gradients of the first and the last
    (batch, head) against the fp64 gradient of that head alone, which
    depends on no other head (Hq = Hkv here)."""
    fa4 = _fa4()
    assert w.Hq == w.Hkv
    q, k, v = workloads.make_inputs(w, seed=0)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa4.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa4.bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    for b, h in ((0, 0), (w.B - 1, w.Hq - 1)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref = ob.attention_bwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(),
                               do[sl].contiguous(), w.scale, w.causal)
        log = [f"{w.name} b={b} h={h}"]
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            _check(name, got[sl], ref[name], log)
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dk.float()).all() \
        and torch.isfinite(dv.float()).all()
