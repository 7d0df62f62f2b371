"""GPU tests of the host-buffer forward (``fa4_fwd_host``): the same bytes
as the device path, argument checks before anything is enqueued, empty
and key-less cases, pageable as well as pinned host memory."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


def _host_out(q):
    B, Sq, Hq, _ = q.shape
    return (torch.full(q.shape, 7.0, dtype=torch.bfloat16).pin_memory(),
            torch.full((B, Hq, Sq), 7.0, dtype=torch.float32).pin_memory())


@pytest.mark.parametrize("case", [(2, 4, 2, 300, 500, 128, True), (1, 2, 2, 256, 256, 64, False)],
                         ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("pinned", [True, False])
def test_host_path_equals_device_path(case, pinned):
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=61)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_ref, lse_ref = fa4.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    o_h, lse_h = _host_out(q)
    ws = torch.empty(fa4.host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream(device=DEV)
    fa4.fwd_host_into(q, k, v, o_h, lse_h, causal, workspace=ws, stream=s)
    s.synchronize()
    assert fa4.device_status(clear=True)[0] == fa4.FA4_OK
    assert torch.equal(o_h, o_ref.cpu()) and torch.equal(lse_h, lse_ref.cpu())


def test_rejected_arguments_enqueue_nothing():
    fa4 = _fa4()
    q, k, v = workloads.make_custom(1, 2, 2, 130, 140, 64, seed=62)
    o_h, lse_h = _host_out(q)
    need = fa4.host_workspace_bytes(1, 2, 2, 130, 140, 64)
    ws = torch.empty(need + 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_host_into(q, k, v, o_h, lse_h, workspace=ws[: need - 1])
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_host_into(q, k, v, o_h, lse_h, workspace=ws[16: 16 + need])
    assert e.value.code == fa4.FA4_ERR_MISALIGNED
    with pytest.raises(fa4.Fa4Error) as e:
        fa4.fwd_host_into(q, k, v, o_h, lse_h, scale=-1.0, workspace=ws)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((o_h == 7.0).all()) and bool((lse_h == 7.0).all())


def test_no_keys_and_no_queries():
    fa4 = _fa4()
    q, _, _ = workloads.make_custom(1, 2, 2, 40, 1, 128, seed=63)
    kv = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16)
    o_h, lse_h = _host_out(q)
    ws = torch.empty(fa4.host_workspace_bytes(1, 2, 2, 40, 0, 128), dtype=torch.uint8, device=DEV)
    fa4.fwd_host_into(q, kv, kv.clone(), o_h, lse_h, workspace=ws)
    torch.cuda.synchronize()
    assert bool((o_h == 0).all()) and bool(torch.isneginf(lse_h).all())
    qe = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16)
    oe, le = torch.empty_like(qe), torch.empty((1, 2, 0), dtype=torch.float32)
    fa4.fwd_host_into(qe, q, q.clone(), oe, le, workspace=ws)
