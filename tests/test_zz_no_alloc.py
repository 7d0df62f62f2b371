"""fa4_fwd_splitkv_static (library-held scratch, no workspace argument)
against fa4_fwd_splitkv with a caller workspace: same kernels, so two
calls in a row must both reproduce it bit for bit. Collected last; it also
passes on its own (the first call sets up the scratch address)."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 2000, 128, True, 4),
                                   (2, 2, 2, 256, 1100, 64, False, 3)],
                         ids=lambda s: "x".join(map(str, s)))
def test_static_scratch_matches_caller_workspace_twice(shape):
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal, splits = shape
    q, k, v = (t.to(DEV) for t in workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=71))
    o_ref, lse_ref = fa4.fwd(q, k, v, causal=causal, num_splits=splits)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        fa4.fwd_splitkv_static_into(q, k, v, o, lse, causal, None, splits)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, detail


def test_static_scratch_rejects_problems_larger_than_it():
    fa4 = _fa4()
    cap = fa4.splitkv_static_max_bytes()
    assert cap == 32 << 20
    # 8 splits x 4096 rows x 16 heads x (128 + 1) fp32 > 32 MiB
    B, Hq, Sq, d, splits = 1, 16, 4096, 128, 8
    assert fa4.splitkv_workspace_bytes(B, Hq, Sq, d, splits) > cap
    q = torch.zeros((B, Sq, Hq, d), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((B, 1024, Hq, d), dtype=torch.bfloat16, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV)
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_splitkv_static_into(q, k, k.clone(), o, lse, False, None, splits)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG


def test_static_scratch_just_under_its_size():
    """A problem whose partial results fill the scratch to within 1 MiB of
    its end: the last split's LSE block sits at the top of the array."""
    fa4 = _fa4()
    cap = fa4.splitkv_static_max_bytes()
    B, Hq, Hkv, Sq, Sk, d, causal, splits = 1, 8, 8, 2000, 2048, 128, False, 4
    need = fa4.splitkv_workspace_bytes(B, Hq, Sq, d, splits)
    assert cap - (1 << 20) < need <= cap
    q, k, v = (t.to(DEV) for t in workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=72))
    o_ref, lse_ref = fa4.fwd(q, k, v, causal=causal, num_splits=splits)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        fa4.fwd_splitkv_static_into(q, k, v, o, lse, causal, None, splits)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, detail


def test_static_scratch_argument_codes_match_the_workspace_entry_point():
    """An unsupported head dimension is reported as such, even when the
    problem would also be too large for the scratch."""
    fa4 = _fa4()
    lib = fa4.load_library()
    B, Hq, Sq, d, splits = 1, 16, 4096, 256, 8
    q = torch.zeros((B, Sq, Hq, d), dtype=torch.bfloat16, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV)
    code = lib.fa4_fwd_splitkv_static(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, Hq, Hq, Sq, Sq, d, 0.0625, 0, splits,
                                      None, None)
    assert code == fa4.FA4_ERR_UNSUPPORTED
