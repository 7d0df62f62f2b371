"""GB300 (sm_103a) fused attention forward: Python binding of ``libfa4.so``.

Every step of the forward pass runs in the library's CUDA kernels; this
module only checks tensor metadata, allocates outputs with torch and
passes pointers to the C ABI declared in ``include/fa4.h``. There is no
CPU or PyTorch fallback: if the library is missing or the device is not an
sm_103 GPU the calls raise.

    o, lse = fwd(q, k, v, causal=True)        # q [B,Sq,Hq,d], k/v [B,Sk,Hkv,d] BF16

The operation is the attention forward of "FlashAttention-4: Algorithm and
Kernel Pipelining Co-Design for Asymmetric Hardware Scaling" (Method,
§3.1): O = softmax(scale * Q K^T [causal mask]) V and the natural-log
LSE per row.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

__all__ = ["fwd", "fwd_into", "fwd_host_into", "host_workspace_bytes", "fwd_fp8", "fwd_fp8_into", "exp2_eval", "device_status", "status_string", "version",
           "lib_path", "load_library", "Fa4Error", "FA4_OK", "FA4_ERR_INVALID_ARG",
           "FA4_ERR_UNSUPPORTED", "FA4_ERR_MISALIGNED", "FA4_ERR_CUDA", "FA4_ERR_TIMEOUT"]

FA4_OK = 0
FA4_ERR_INVALID_ARG = 1
FA4_ERR_UNSUPPORTED = 2
FA4_ERR_MISALIGNED = 3
FA4_ERR_CUDA = 4
FA4_ERR_TIMEOUT = 5

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libfa4.so")
_lib = None


class Fa4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code) if _lib else code}")


class _Options(ctypes.Structure):
    _fields_ = [("tau", ctypes.c_float), ("exp2_emulation", ctypes.c_int),
                ("rescale_stats", ctypes.c_void_p), ("trace", ctypes.c_void_p),
                ("trace_ctas", ctypes.c_int), ("strict_mma_order", ctypes.c_int),
                ("grid_mode", ctypes.c_int), ("correction_warpgroup", ctypes.c_int),
                ("test_stall_cycles", ctypes.c_longlong)]


class _BwdOptions(ctypes.Structure):
    """fa4_bwd_options (include/fa4.h)."""
    _fields_ = [("deterministic", ctypes.c_int), ("test_stall_cycles", ctypes.c_longlong)]


TRACE_EVENTS = 21
TRACE_STEPS = 128
TRACE_EVENT_NAMES = ("mma_s_wait", "mma_s_issued", "mma_pv_wait", "mma_pv_issued",
                     "sm_s_ready", "sm_loaded", "sm_exp_done", "sm_arrived",
                     "co_wake", "co_arrived", "mma_s_go", "mma_pv_go", "sm_arrived_q1",
                     "sm_arrived_q2", "sm_arrived_q3", "sm_max_done",
                     "mma_committed", "mma_v_ready", "load_issued", "sm_max_loop",
                     "sm_c_done")


def load_library():
    """Load ``libfa4.so`` (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(lib_path):
        raise RuntimeError(f"{lib_path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(lib_path)
    vp, i32, f32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
    lib.fa4_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]
    lib.fa4_fwd.restype = i32
    lib.fa4_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                               ctypes.POINTER(_Options), vp]
    lib.fa4_fwd_ex.restype = i32
    lib.fa4_fwd_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.fa4_fwd_host_workspace_bytes.restype = ctypes.c_uint64
    lib.fa4_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp,
                                 ctypes.c_uint64, vp, vp]
    lib.fa4_fwd_host.restype = i32
    lib.fa4_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                f32, f32, f32, vp, vp]
    lib.fa4_fwd_fp8.restype = i32
    lib.fa4_fwd_splitkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.fa4_fwd_splitkv_workspace_bytes.restype = ctypes.c_uint64
    lib.fa4_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                    i32, vp, ctypes.c_uint64, ctypes.POINTER(_Options), vp]
    lib.fa4_fwd_splitkv.restype = i32
    lib.fa4_fwd_splitkv_static_max_bytes.argtypes = []
    lib.fa4_fwd_splitkv_static_max_bytes.restype = ctypes.c_uint64
    lib.fa4_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                           i32, i32, ctypes.POINTER(_Options), vp]
    lib.fa4_fwd_splitkv_static.restype = i32
    lib.fa4_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.fa4_bwd_workspace_bytes.restype = ctypes.c_uint64
    lib.fa4_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                            vp, ctypes.c_uint64, vp]
    lib.fa4_bwd.restype = i32
    lib.fa4_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                               i32, i32, vp, ctypes.c_uint64, vp]
    lib.fa4_bwd_ex.restype = i32
    lib.fa4_bwd_default_options.argtypes = [ctypes.POINTER(_BwdOptions)]
    lib.fa4_bwd_default_options.restype = None
    lib.fa4_bwd_opt.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                i32, ctypes.POINTER(_BwdOptions), vp, ctypes.c_uint64, vp]
    lib.fa4_bwd_opt.restype = i32
    lib.fa4_fwd_default_options.argtypes = [ctypes.POINTER(_Options)]
    lib.fa4_fwd_default_options.restype = None
    lib.fa4_device_status.argtypes = [i32, ctypes.POINTER(ctypes.c_uint * 4)]
    lib.fa4_device_status.restype = i32
    lib.fa4_exp2_eval.argtypes = [vp, vp, vp, i64, vp]
    lib.fa4_exp2_eval.restype = i32
    lib.fa4_status_string.argtypes = [i32]
    lib.fa4_status_string.restype = ctypes.c_char_p
    lib.fa4_version.argtypes = []
    lib.fa4_version.restype = i32
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().fa4_status_string(int(code)).decode()


def version() -> int:
    return int(load_library().fa4_version())


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check(code: int, what: str) -> None:
    if code != FA4_OK:
        raise Fa4Error(code, what)


def fwd_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, causal: bool = False, scale: Optional[float] = None, *,
             tau: float = 8.0, exp2_emulation: int = 0,
             rescale_stats: Optional[torch.Tensor] = None,
             trace: Optional[torch.Tensor] = None, strict_mma_order: bool = False,
             grid_mode: int = 0, num_splits: int = 0,
             workspace: Optional[torch.Tensor] = None, correction_warpgroup: bool = False,
             test_stall_cycles: int = 0,
             stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write attention forward into preallocated ``o`` and ``lse``.

    Shapes: q, o [B,Sq,Hq,d]; k, v [B,Sk,Hkv,d] (BF16, contiguous, CUDA);
    lse [B,Hq,Sq] fp32. ``scale`` defaults to 1/sqrt(d). ``num_splits`` > 0
    runs the key-range split forward (``fa4_fwd_splitkv``) with
    ``workspace`` (a CUDA uint8 tensor of at least
    ``splitkv_workspace_bytes(...)`` bytes; allocated here when omitted).
    """
    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,Sq,Hq,d] and k, v [B,Sk,Hkv,d]")
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("o must match q and lse must be [B,Hq,Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    opt = _Options()
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    opt.tau = float(tau)
    # True / False are accepted as 8 / 0 (one entry pair in 8 / none)
    emu = 8 if exp2_emulation is True else int(exp2_emulation)
    if emu not in (0, 4, 8):
        raise ValueError("exp2_emulation must be 0, 4 or 8 (or a bool)")
    opt.exp2_emulation = emu
    opt.strict_mma_order = 1 if strict_mma_order else 0
    opt.grid_mode = int(grid_mode)
    opt.test_stall_cycles = int(test_stall_cycles)
    opt.correction_warpgroup = 1 if correction_warpgroup else 0
    if rescale_stats is not None:
        if rescale_stats.dtype != torch.int64 or rescale_stats.numel() < 2 or not rescale_stats.is_cuda:
            raise ValueError("rescale_stats must be a CUDA int64 tensor of 2 elements")
        opt.rescale_stats = rescale_stats.data_ptr()
    if trace is not None:
        per_cta = TRACE_EVENTS * TRACE_STEPS * 2
        if trace.dtype != torch.int64 or not trace.is_cuda or trace.numel() % per_cta:
            raise ValueError("trace must be a CUDA int64 tensor of n_ctas * "
                             f"{per_cta} elements")
        opt.trace = trace.data_ptr()
        opt.trace_ctas = trace.numel() // per_cta
    if num_splits:
        need = splitkv_workspace_bytes(B, Hq, Sq, d, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
        code = lib.fa4_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, Hq, Hkv, Sq, Sk, d, float(scale),
                                   int(bool(causal)), int(num_splits), workspace.data_ptr(),
                                   workspace.numel(), ctypes.byref(opt), _stream_handle(stream))
        _check(code, "fa4_fwd_splitkv")
        return
    code = lib.fa4_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, Hq, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                          ctypes.byref(opt), _stream_handle(stream))
    _check(code, "fa4_fwd_ex")


def fwd_splitkv_static_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                            lse: torch.Tensor, causal: bool, scale: Optional[float],
                            num_splits: int, stream: Optional[torch.cuda.Stream] = None) -> None:
    """``fa4_fwd_splitkv_static``: the key-range split forward with the
    library's own fixed device scratch (no workspace argument). Same tensor
    rules as ``fwd_into``; default options."""
    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Sq) or v.shape != k.shape:
        raise ValueError("o must match q, v must match k and lse must be [B,Hq,Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = lib.fa4_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, Hq, Hkv, Sq, Sk, d, float(scale),
                                      int(bool(causal)), int(num_splits), None,
                                      _stream_handle(stream))
    _check(code, "fa4_fwd_splitkv_static")


def splitkv_static_max_bytes() -> int:
    """Size of the library-held scratch of ``fwd_splitkv_static_into``."""
    return int(load_library().fa4_fwd_splitkv_static_max_bytes())


def bwd_workspace_bytes(B: int, Hq: int, Sq: int, d: int) -> int:
    """Device scratch bytes the backward needs."""
    return int(load_library().fa4_bwd_workspace_bytes(B, Hq, Sq, d))


def bwd_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             dout: torch.Tensor, lse: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
             dv: torch.Tensor, causal: bool = False, scale: Optional[float] = None, *,
             deterministic: bool = False, test_stall_cycles: int = 0,
             workspace: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> None:
    """``fa4_bwd_opt``: write dq, dk, dv (preallocated, BF16) for the upstream
    gradient ``dout``; ``o`` and ``lse`` are the forward's outputs.
    ``workspace`` (CUDA uint8) is allocated here when omitted.
    ``test_stall_cycles`` > 0 is a diagnostic that makes the launch time out."""
    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("dout", dout, torch.bfloat16), ("lse", lse, torch.float32),
                        ("dq", dq, torch.bfloat16), ("dk", dk, torch.bfloat16),
                        ("dv", dv, torch.bfloat16)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if (o.shape != q.shape or dout.shape != q.shape or dq.shape != q.shape or v.shape != k.shape
            or dk.shape != k.shape or dv.shape != k.shape or tuple(lse.shape) != (B, Hq, Sq)):
        raise ValueError("shapes: q, o, dout, dq [B,Sq,Hq,d]; k, v, dk, dv [B,Sk,Hkv,d]; "
                         "lse [B,Hq,Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bwd_workspace_bytes(B, Hq, Sq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    opt = _BwdOptions()
    lib.fa4_bwd_default_options(ctypes.byref(opt))
    opt.deterministic = int(bool(deterministic))
    opt.test_stall_cycles = int(test_stall_cycles)
    code = lib.fa4_bwd_opt(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                           lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv,
                           Sq, Sk, d, float(scale), int(bool(causal)), ctypes.byref(opt),
                           workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(code, "fa4_bwd_opt")


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
        lse: torch.Tensor, causal: bool = False, scale: Optional[float] = None, **kw
        ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Attention backward; returns (dq, dk, dv)."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bwd_into(q, k, v, o, dout, lse, dq, dk, dv, causal, scale, **kw)
    return dq, dk, dv


def host_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int) -> int:
    """Device scratch bytes ``fwd_host_into`` needs."""
    return int(load_library().fa4_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d))


def fwd_host_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                  lse: torch.Tensor, causal: bool = False, scale: Optional[float] = None, *,
                  workspace: torch.Tensor, tau: float = 8.0, exp2_emulation: int = 0,
                  grid_mode: int = 0, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Forward on HOST tensors (``fa4_fwd_host``): q, k, v, o, lse are CPU
    tensors (pinned for asynchronous copies) with the layouts of ``fwd_into``;
    ``workspace`` is a CUDA uint8 tensor of ``host_workspace_bytes(...)``
    bytes. The copies and the forward are enqueued on ``stream``; o and lse
    hold the result once the stream has passed the call."""
    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,Sq,Hq,d] and k, v [B,Sk,Hkv,d]")
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("o must match q and lse must be [B,Hq,Sq]")
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    opt = _Options()
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    opt.tau = float(tau)
    emu = 8 if exp2_emulation is True else int(exp2_emulation)
    if emu not in (0, 4, 8):
        raise ValueError("exp2_emulation must be 0, 4 or 8 (or a bool)")
    opt.exp2_emulation = emu
    opt.grid_mode = int(grid_mode)
    code = lib.fa4_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, Hq, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                            workspace.data_ptr(), workspace.numel(), ctypes.byref(opt),
                            _stream_handle(stream))
    _check(code, "fa4_fwd_host")


def fwd_fp8_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                 lse: torch.Tensor, q_scale: float, k_scale: float, v_scale: float,
                 causal: bool = False, scale: Optional[float] = None, *, tau: float = 8.0,
                 rescale_stats: Optional[torch.Tensor] = None,
                 strict_mma_order: bool = False, grid_mode: int = 0,
                 correction_warpgroup: bool = False,
                 stream: Optional[torch.cuda.Stream] = None) -> None:
    """FP8 forward (``fa4_fwd_fp8``) into preallocated ``o`` and ``lse``.

    q [B,Sq,Hq,128], k/v [B,Sk,Hkv,128] hold e4m3 codes (torch.float8_e4m3fn,
    or uint8 bit patterns) whose true values are code * q_scale / k_scale /
    v_scale; o [B,Sq,Hq,128] BF16 and lse [B,Hq,Sq] fp32 receive the forward
    of the true values. ``scale`` defaults to 1/sqrt(128).
    """
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must be float8_e4m3fn (or uint8 codes), got {t.dtype}")
    for name, t, dt in (("o", o, torch.bfloat16), ("lse", lse, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,Sq,Hq,d] and k, v [B,Sk,Hkv,d]")
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("o must match q and lse must be [B,Hq,Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    opt = _Options()
    lib.fa4_fwd_default_options(ctypes.byref(opt))
    opt.tau = float(tau)
    opt.strict_mma_order = 1 if strict_mma_order else 0
    opt.grid_mode = int(grid_mode)
    opt.correction_warpgroup = 1 if correction_warpgroup else 0
    if rescale_stats is not None:
        if rescale_stats.dtype != torch.int64 or rescale_stats.numel() < 2 or not rescale_stats.is_cuda:
            raise ValueError("rescale_stats must be a CUDA int64 tensor of 2 elements")
        opt.rescale_stats = rescale_stats.data_ptr()
    code = lib.fa4_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, Hq, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                           float(q_scale), float(k_scale), float(v_scale), ctypes.byref(opt),
                           _stream_handle(stream))
    _check(code, "fa4_fwd_fp8")


def fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_scale: float, k_scale: float,
            v_scale: float, causal: bool = False, scale: Optional[float] = None,
            **kw) -> Tuple[torch.Tensor, torch.Tensor]:
    """FP8 forward; returns (o [B,Sq,Hq,128] BF16, lse [B,Hq,Sq] fp32)."""
    B, Sq, Hq, d = q.shape
    o = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    fwd_fp8_into(q, k, v, o, lse, q_scale, k_scale, v_scale, causal, scale, **kw)
    return o, lse


def splitkv_workspace_bytes(B: int, Hq: int, Sq: int, d: int, num_splits: int) -> int:
    """Device scratch bytes the key-range split forward needs."""
    return int(load_library().fa4_fwd_splitkv_workspace_bytes(B, Hq, Sq, d, num_splits))


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: Optional[float] = None, **kw) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention forward; returns (o [B,Sq,Hq,d] BF16, lse [B,Hq,Sq] fp32)."""
    B, Sq, Hq, _ = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    fwd_into(q, k, v, o, lse, causal, scale, **kw)
    return o, lse


def exp2_eval(x: torch.Tensor, stream: Optional[torch.cuda.Stream] = None
              ) -> Tuple[torch.Tensor, torch.Tensor]:
    """The kernel's two 2^x paths on fp32 CUDA input: (emulated, MUFU.EX2)."""
    lib = load_library()
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    y_emu = torch.empty_like(x)
    y_mufu = torch.empty_like(x)
    _check(lib.fa4_exp2_eval(x.data_ptr(), y_emu.data_ptr(), y_mufu.data_ptr(), x.numel(),
                             _stream_handle(stream)), "fa4_exp2_eval")
    return y_emu, y_mufu


def device_status(clear: bool = True) -> Tuple[int, Tuple[int, int, int, int]]:
    """Synchronise and read the kernels' status word: (code, detail[4])."""
    lib = load_library()
    detail = (ctypes.c_uint * 4)()
    code = lib.fa4_device_status(1 if clear else 0, ctypes.byref(detail))
    return int(code), tuple(int(x) for x in detail)
