"""The C-ABI library loads without a GPU, exports every function that
include/fa4.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attention_forward_fa4_gb300 import build
    build.build()
    import attention_forward_fa4_gb300 as fa4
    return fa4.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "fa4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa4_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "fa4_fwd" in names and "fa4_fwd_ex" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for code, name in enumerate(["FA4_OK", "FA4_ERR_INVALID_ARG", "FA4_ERR_UNSUPPORTED",
                                 "FA4_ERR_MISALIGNED", "FA4_ERR_CUDA", "FA4_ERR_TIMEOUT"]):
        assert lib.fa4_status_string(code).decode() == name
    assert lib.fa4_version() >= 100


P = 0x100000          # aligned stand-in addresses: never dereferenced on failure paths
Q, K, V, O, L = P, 2 * P, 3 * P, 4 * P, 5 * P


def _call(lib, q=Q, k=K, v=V, o=O, lse=L, B=1, Hq=2, Hkv=2, Sq=64, Sk=64, d=64, scale=0.125,
          causal=0):
    return lib.fa4_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, None)


def test_argument_errors_launch_nothing(lib):
    import attention_forward_fa4_gb300 as fa4
    assert _call(lib, q=0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, o=0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, lse=0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, k=0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, Hq=3, Hkv=2) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, Hkv=0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, B=-1) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, Sk=-5) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, scale=0.0) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, scale=float("nan")) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, causal=2) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, d=96) == fa4.FA4_ERR_UNSUPPORTED
    assert _call(lib, d=256) == fa4.FA4_ERR_UNSUPPORTED
    assert _call(lib, q=Q + 8) == fa4.FA4_ERR_MISALIGNED
    assert _call(lib, v=V + 2) == fa4.FA4_ERR_MISALIGNED
    assert _call(lib, lse=L + 2) == fa4.FA4_ERR_MISALIGNED
    # o overlapping q, lse overlapping v
    assert _call(lib, o=Q + 16) == fa4.FA4_ERR_INVALID_ARG
    assert _call(lib, lse=V) == fa4.FA4_ERR_INVALID_ARG


def test_empty_problems_are_no_ops(lib):
    import attention_forward_fa4_gb300 as fa4
    assert _call(lib, B=0, q=0, k=0, v=0, o=0, lse=0) == fa4.FA4_OK
    assert _call(lib, Sq=0, q=0, o=0, lse=0) == fa4.FA4_OK


def test_options_are_validated(lib):
    import attention_forward_fa4_gb300 as fa4
    from attention_forward_fa4_gb300 import _Options
    opt = _Options()
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    assert opt.tau == 8.0 and opt.exp2_emulation == 0 and not opt.rescale_stats
    for tau in (-1.0, float("inf"), 100.0):
        opt.tau = tau
        assert lib.fa4_fwd_ex(Q, K, V, O, L, 1, 2, 2, 64, 64, 64, 0.125, 0, ctypes.byref(opt),
                              None) == fa4.FA4_ERR_INVALID_ARG
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    opt.exp2_emulation = 3
    assert lib.fa4_fwd_ex(Q, K, V, O, L, 1, 2, 2, 64, 64, 64, 0.125, 0, ctypes.byref(opt),
                          None) == fa4.FA4_ERR_INVALID_ARG


def test_without_a_device_valid_calls_report_cuda_error(lib):
    import torch
    import attention_forward_fa4_gb300 as fa4
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib) in (fa4.FA4_ERR_CUDA, fa4.FA4_ERR_UNSUPPORTED)


def test_trace_layout_matches_header():
    import attention_forward_fa4_gb300 as fa4
    hdr = open(os.path.join(ROOT, "include", "fa4.h")).read()
    n_ev = int(re.search(r"#define FA4_TRACE_EVENTS (\d+)", hdr).group(1))
    n_st = int(re.search(r"#define FA4_TRACE_STEPS (\d+)", hdr).group(1))
    assert fa4.TRACE_EVENTS == n_ev == len(fa4.TRACE_EVENT_NAMES)
    assert fa4.TRACE_STEPS == n_st


def test_fp8_and_host_entry_points_check_arguments_first(lib):
    """fa4_fwd_fp8 and fa4_fwd_host reject bad arguments before any CUDA
    call (so the same codes come back with and without a GPU)."""
    import attention_forward_fa4_gb300 as fa4
    f32 = ctypes.c_float

    def fp8(d=128, qs=1.0, ks=1.0, vs=1.0, q=Q):
        return lib.fa4_fwd_fp8(q, K, V, O, L, 1, 2, 2, 64, 64, d, 0.125, 0, f32(qs), f32(ks),
                               f32(vs), None, None)

    assert fp8(qs=0.0) == fa4.FA4_ERR_INVALID_ARG
    assert fp8(vs=float("inf")) == fa4.FA4_ERR_INVALID_ARG
    assert fp8(ks=-1.0) == fa4.FA4_ERR_INVALID_ARG
    assert fp8(d=64) == fa4.FA4_ERR_UNSUPPORTED
    assert fp8(q=Q + 8) == fa4.FA4_ERR_MISALIGNED
    from attention_forward_fa4_gb300 import _Options
    opt = _Options()
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    opt.exp2_emulation = 8
    assert lib.fa4_fwd_fp8(Q, K, V, O, L, 1, 2, 2, 64, 64, 128, 0.125, 0, f32(1.0), f32(1.0),
                           f32(1.0), ctypes.byref(opt), None) == fa4.FA4_ERR_UNSUPPORTED

    need = lib.fa4_fwd_host_workspace_bytes(1, 2, 2, 64, 80, 64)
    # q, o: 16 KB each; k, v: 20 KB each; lse 512 B -> each rounded up to 256 B
    assert need == 2 * 16384 + 2 * 20480 + 512
    assert lib.fa4_fwd_host_workspace_bytes(1, 2, 2, 64, 80, 96) == 0
    W = 8 * P

    def host(ws=W, ws_bytes=need, d=64, B=1, q=Q, scale=0.125):
        return lib.fa4_fwd_host(q, K, V, O, L, B, 2, 2, 64, 80, d, scale, 0, ws, ws_bytes, None,
                                None)

    assert host(ws=0) == fa4.FA4_ERR_INVALID_ARG
    assert host(ws_bytes=need - 1) == fa4.FA4_ERR_INVALID_ARG
    assert host(ws=W + 128) == fa4.FA4_ERR_MISALIGNED
    assert host(d=96) == fa4.FA4_ERR_UNSUPPORTED
    assert host(B=-1) == fa4.FA4_ERR_INVALID_ARG
    assert host(q=0) == fa4.FA4_ERR_INVALID_ARG
    assert host(scale=-1.0) == fa4.FA4_ERR_INVALID_ARG
    assert host(B=0) == fa4.FA4_OK        # empty: nothing to copy or compute


def test_bwd_options_are_checked_before_cuda(lib):
    """fa4_bwd_opt rejects a deterministic flag outside {0, 1} and a negative
    diagnostic stall before any device call; the defaults are off."""
    import attention_forward_fa4_gb300 as fa4
    opt = fa4._BwdOptions()
    lib.fa4_bwd_default_options(ctypes.byref(opt))
    assert opt.deterministic == 0 and opt.test_stall_cycles == 0
    P = 1 << 20       # 16-byte aligned fake device addresses: never dereferenced here

    def call(o):
        return lib.fa4_bwd_opt(P, P + 4096, P + 8192, P + 12288, P + 16384, P + 20480, P + 24576,
                               P + 28672, P + 32768, 1, 2, 2, 64, 64, 64, 0.125, 0,
                               ctypes.byref(o), P + 65536, 1 << 20, None)
    bad = fa4._BwdOptions(deterministic=2, test_stall_cycles=0)
    assert call(bad) == fa4.FA4_ERR_INVALID_ARG
    bad = fa4._BwdOptions(deterministic=0, test_stall_cycles=-1)
    assert call(bad) == fa4.FA4_ERR_INVALID_ARG
