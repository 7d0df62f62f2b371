"""The kernels' timeout path, exercised without a GPU fault.

Every pipeline wait in the forward kernel is bounded; when one runs out the
CTA raises its abort flag, records (code, role, barrier, block) in the
device status word, drains its in-flight copies and MMAs, frees tensor
memory and exits. The diagnostic option ``test_stall_cycles`` makes the
softmax warps wait on a barrier that nothing completes, with that many
cycles as their limit, so this path runs on a normal launch. The context
must stay usable: the next launch on it matches the oracle.
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
