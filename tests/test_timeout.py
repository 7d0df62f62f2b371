"""The kernels' timeout path, exercised without a GPU fault.

Every pipeline wait in the forward and backward kernels is bounded; when one
runs out the CTA raises its abort flag, records (code, role, barrier, block)
in the device status word, drains its in-flight copies and MMAs, frees
tensor memory and exits. The diagnostic option ``test_stall_cycles`` makes
the softmax warps (forward) or the compute warps (backward) wait on a
barrier that nothing completes, with that many cycles as their limit, so
this path runs on a normal launch. The context must stay usable: the next
launch on it matches the oracle.
"""
import math

import pytest
import torch

import workloads
from oracle import attn as oracle
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FA4_ERR_TIMEOUT = 5
ROLE_SOFTMAX = 2


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


@pytest.mark.parametrize("shape", [(1, 4, 4, 512, 512, 128, True), (2, 2, 2, 300, 700, 64, False)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("grid_mode", [1, 2])
def test_stalled_wait_times_out_and_the_context_recovers(shape, grid_mode):
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=81)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    fa4.device_status(clear=True)
    o = torch.full((B, Sq, Hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, Hq, Sq), 7.0, dtype=torch.float32, device=DEV)
    fa4.fwd_into(qd, kd, vd, o, lse, causal, None, grid_mode=grid_mode, test_stall_cycles=20000)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == FA4_ERR_TIMEOUT, (code, detail)
    assert detail[0] == FA4_ERR_TIMEOUT and detail[1] == ROLE_SOFTMAX
    n_tiles = B * Hq * math.ceil(Sq / 256)
    assert 0 <= detail[3] < n_tiles
    # the epilogue never ran: the outputs keep their fill
    assert (o == 7.0).all() and (lse == 7.0).all()
    # the status word was cleared, and the same context computes correctly
    code, _ = fa4.device_status(clear=False)
    assert code == fa4.FA4_OK
    o2, lse2 = fa4.fwd(qd, kd, vd, causal=causal, grid_mode=grid_mode)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, detail
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 1.0 / math.sqrt(d), causal)
    parity.assert_close(parity.to_np(o2), parity.to_np(lse2), o_ref, lse_ref, "after timeout")


def test_negative_stall_is_rejected():
    fa4 = _fa4()
    q, k, v = (t.to(DEV) for t in workloads.make_custom(1, 2, 2, 64, 64, 64, seed=82))
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd(q, k, v, test_stall_cycles=-1)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(1, 4, 2, 512, 512, 128, True), (2, 2, 2, 300, 700, 64, False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_backward_stalled_wait_times_out_and_the_context_recovers(shape):
    """The same for the backward: every role of every CTA leaves through its
    abort path (load drains its copies, the MMA warp its MMAs, the flush warp
    its reduce-adds), dK and dV are not written, and the next backward on
    the context matches the fp64 gradient."""
    from oracle import attn_bwd as ob
    from tests.test_bwd_parity import _check
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=83)
    do = torch.randn((B, Sq, Hq, d), generator=torch.Generator().manual_seed(84)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa4.fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa4.device_status(clear=True)
    dq = torch.empty_like(qd)
    dk = torch.full_like(kd, 7.0)
    dv = torch.full_like(vd, 7.0)
    fa4.bwd_into(qd, kd, vd, o, dod, lse, dq, dk, dv, causal, scale, test_stall_cycles=20000)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == FA4_ERR_TIMEOUT, (code, detail)
    assert detail[0] == FA4_ERR_TIMEOUT and detail[1] == ROLE_SOFTMAX
    n_ctas = B * Hkv * math.ceil(Sk / 128)
    assert 0 <= detail[3] < n_ctas
    # no epilogue ran: dk and dv keep their fill
    assert (dk == 7.0).all() and (dv == 7.0).all()
    code, _ = fa4.device_status(clear=False)
    assert code == fa4.FA4_OK
    dq2, dk2, dv2 = fa4.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, detail
    ref = ob.attention_bwd(q, k, v, do, scale, causal)
    log = [f"after timeout {shape}"]
    for name, got in (("dq", dq2), ("dk", dk2), ("dv", dv2)):
        _check(name, got, ref[name], log)


def test_backward_negative_stall_is_rejected():
    fa4 = _fa4()
    q, k, v = (t.to(DEV) for t in workloads.make_custom(1, 2, 2, 64, 64, 64, seed=85))
    o, lse = fa4.fwd(q, k, v)
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.bwd(q, k, v, o, torch.ones_like(q), lse, test_stall_cycles=-1)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
