"""GPU parity of the key-range split forward (fa4_fwd_splitkv) against the
fp64 definition, its per-split partials against the key-range model, and
its argument checks. Every call goes through the C ABI."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn as oracle
from oracle import splitkv as sk
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fa4():
    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()
    return fa4


def _run(q, k, v, causal, splits, scale=None, workspace=None, **kw):
    fa4 = _fa4()
    o, lse = fa4.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale,
                     num_splits=splits, workspace=workspace, **kw)
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    assert code == fa4.FA4_OK, f"device status {code} {detail}"
    return o, lse


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal, splits
    (1, 2, 2, 256, 1024, 128, False, 4),
    (1, 2, 2, 256, 1024, 128, True, 3),
    (2, 4, 2, 200, 1000, 64, True, 5),      # GQA, ragged Sq and Sk, bottom-right causal
    (1, 8, 8, 128, 2500, 128, False, 7),    # ragged last block
    (1, 2, 1, 700, 300, 64, True, 2),       # Sq > Sk: leading rows see no key
    (3, 2, 2, 129, 257, 128, True, 1),      # one split: same path, one range
    (1, 2, 2, 64, 512, 64, False, 16),      # more splits than blocks: 4 ranges
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_splitkv_matches_oracle(case):
    B, Hq, Hkv, Sq, Sk, d, causal, splits = case
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=51)
    o, lse = _run(q, k, v, causal, splits)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 1.0 / math.sqrt(d), causal)
    parity.assert_close(parity.to_np(o), parity.to_np(lse), o_ref, lse_ref, str(case))


def test_partials_match_the_key_range_model():
    """The workspace holds each split's normalised O_s and LSE_s (layout of
    include/fa4.h); compare them with the fp64 key-range forward."""
    fa4 = _fa4()
    B, Hq, Hkv, Sq, Sk, d, causal, splits = 1, 4, 2, 300, 900, 64, True, 3
    q, k, v = workloads.make_custom(B, Hq, Hkv, Sq, Sk, d, seed=52)
    need = fa4.splitkv_workspace_bytes(B, Hq, Sq, d, splits)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    _run(q, k, v, causal, splits, workspace=ws)
    f = ws.view(torch.float32).cpu().numpy().astype(np.float64)
    n_o = splits * B * Sq * Hq * d
    o_part = f[:n_o].reshape(splits, B, Sq, Hq, d)
    lse_part = f[n_o:n_o + splits * B * Hq * Sq].reshape(splits, B, Hq, Sq)
    ranges = sk.split_ranges(Sk, splits)
    assert len(ranges) == splits
    for s, (k0, k1) in enumerate(ranges):
        o_ref, lse_ref = sk.keyrange_fwd(q, k, v, 1.0 / math.sqrt(d), causal, k0, k1)
        assert np.abs(o_part[s] - o_ref).max() <= 2e-2, s
        fin = np.isfinite(lse_ref)
        assert (np.isneginf(lse_part[s]) == ~fin).all(), s
        assert np.abs(lse_part[s][fin] - lse_ref[fin]).max() <= 1e-3, s


def test_long_keys_sampled_rows_and_agreement_with_unsplit():
    w = workloads.Workload("split_long", 1, 8, 2, 512, 32768, 128, True)
    q, k, v = workloads.make_inputs(w, seed=0)
    o, lse = _run(q, k, v, True, 32)
    rows = workloads.sample_rows(w, n_random=256, seed=2, edge=16, max_bh=8)
    o_ref, lse_ref = oracle.attention_fwd_rows(q, k, v, w.scale, True, rows)
    o_g, l_g = parity.gather_gpu_rows(o, lse, rows)
    parity.assert_close(o_g, l_g, o_ref, lse_ref, w.name)
    o1, l1 = _run(q, k, v, True, 0)             # the plain forward
    assert (o.float() - o1.float()).abs().max().item() <= 2e-2
    assert (lse - l1).abs().max().item() <= 1e-3


def test_workspace_and_split_count_are_checked():
    fa4 = _fa4()
    q, k, v = workloads.make_custom(1, 2, 2, 64, 512, 64, seed=53)
    need = fa4.splitkv_workspace_bytes(1, 2, 64, 64, 4)
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa4.Fa4Error) as e:
        _run(q, k, v, False, 4, workspace=small)
    assert e.value.code == fa4.FA4_ERR_INVALID_ARG
    for bad in (-1, 129):
        with pytest.raises(fa4.Fa4Error):
            _run(q, k, v, False, bad)
    ws = torch.empty(need + 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa4.Fa4Error) as e:
        _run(q, k, v, False, 4, workspace=ws[1:])          # misaligned
    assert e.value.code == fa4.FA4_ERR_MISALIGNED
