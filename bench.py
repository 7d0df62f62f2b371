"""Benchmark of the GB300 attention forward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--tau T] [--exp2-emulation 0|4|8]
                    [--pass fwd|bwd] [--num-splits S] [--precision bf16|fp8]

One step = one attention forward over the workload's synthetic BF16 input
(default: B=2, Hq=Hkv=16, Sq=Sk=8192, d=128, causal). ``value`` is the
whole-job TFLOP/s (4*B*Hq*Sq*Sk*d, halved for causal) from CUDA events
around each launch, with the inputs resident in HBM and L2 flushed before
every timed launch. ``e2e`` is the same metric with the host->device copy
of q, k, v and the device->host copy of o and lse inside each step.

Under torchrun (N > 1) each rank runs its own shard of a global batch
(weak scaling, no collective on the data path); time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead
(rank 0 only), each step a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time
from typing import Dict, List, Optional, Tuple

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s on 1 GB300 (BF16) and % of 2.25 PFLOP/s roofline"
METRIC_BWD = ("attention bwd TFLOP/s (2.5 x forward FLOPs: five products) on 1 GB300 (BF16) "
              "and % of 2.25 PFLOP/s roofline")
METRIC_FP8 = ("attention fwd TFLOP/s on 1 GB300 (FP8 e4m3 Q, K, V and P, BF16 O) and % of "
              "4.5 PFLOP/s roofline")
BWD_FLOP_FACTOR = 2.5
FP8_OVER_BF16 = 2.0            # nominal dense FP8 : BF16 tensor rate (4.5 / 2.25 PFLOP/s)
NOMINAL_BF16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_NAME = "fa4_fwd_kernel"


# ---------------------------------------------------------------- helpers
def dist_env() -> Tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_workload(w: workloads.Workload, rank: int, world: int) -> Tuple[workloads.Workload, int]:
    """Weak scaling: every rank owns B batches of a global batch of B*world.

    Returns the per-rank workload and the batch offset of its shard (used to
    seed distinct data per shard)."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad rank/world")
    return w, rank * w.B


def max_over_ranks(values: List[float], dist, device) -> List[float]:
    """Element-wise max of per-rank timings (the job is as slow as its
    slowest rank)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# Source files each kernel's code and launch depend on.
KERNEL_SOURCES = {
    "fa4_fwd_kernel": ["fa4_fwd_kernel.cuh", "fa4_ptx.cuh", "fa4_exp2.cuh", "fa4_launch.cuh",
                       "fa4_internal.h", "fa4_api.cu", "fa4_fwd_d128.cu", "fa4_fwd_d64.cu",
                       "fa4_fwd_fp8.cu", "fa4_merge.cu"],
    "fa4_bwd_kernel": ["fa4_bwd_q64.cuh", "fa4_bwd.cu", "fa4_fwd_kernel.cuh", "fa4_ptx.cuh",
                       "fa4_exp2.cuh", "fa4_internal.h", "fa4_api.cu"],
}


def kernel_sources_hash(kernel: str = KERNEL_NAME) -> str:
    """Hash of the sources a kernel depends on; a stored ncu traffic figure
    only applies to the build it was measured on."""
    csrc = os.path.join(ROOT, "attention_forward_fa4_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(workload_name: str, kernel: str = KERNEL_NAME) -> Optional[dict]:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_sources_hash:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_sources_hash(kernel):
        return None
    return {"bytes": float(m_b.group(1)), "source": os.path.relpath(path, ROOT)}


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "_source": "fallback"}


def fp8_gemm_peak_tflops(dev) -> Optional[float]:
    """Burst rate of a dense e4m3 GEMM (torch._scaled_mm, cuBLASLt) at
    8192^3 on this GPU: the FP8 counterpart of MEASURED_PEAKS' BF16 figure.
    Best of 10 timed calls after 3 warm-ups; None if the call is unavailable."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        def fn():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record()
            fn()
            s1.record()
            torch.cuda.synchronize()
            best = min(best, s0.elapsed_time(s1))
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def table1_cycles(M: int, N: int, d: int, flops_per_clk: float = 8192.0,
                  exp_per_clk: float = 16.0, smem_bytes_per_clk: float = 128.0) -> dict:
    """Closed-form forward roofline per key block ("FlashAttention-4", Table 1,
    §3.1.1): MMA = 4*M*N*d / F; exp = M*N / MUFU rate; SMEM = bytes of the
    operands read from shared memory by the MMAs / SMEM bandwidth. Each
    128-row slice of the M rows reads Q, K and V (N x d BF16 each)."""
    mma = 4.0 * M * N * d / flops_per_clk
    exp = M * N / exp_per_clk
    smem = (M // 128) * 3 * N * d * 2 / smem_bytes_per_clk
    return {"mma": mma, "exp": exp, "smem": smem}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self, t0: float, t1: float) -> Optional[dict]:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5], parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        if not inside:
            return None
        sm = sorted(r[1] for r in inside)
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for name, flag in zip(names, r[4]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------- CPU oracle leg
def oracle_rate(w: workloads.Workload, q, k, v, seconds: float, seed: int = 0,
                scale: Optional[float] = None) -> Tuple[float, float, int, str]:
    """Time the fp64 oracle on a seeded random row sample sized for about
    ``seconds`` of host work; returns (flop/s, flops done, threads, sample)."""
    scale = w.scale if scale is None else scale
    import numpy as np
    from oracle import attn as oracle

    def flops_of(rows):
        i = rows % w.Sq
        keys = np.minimum(w.Sk, i + (w.Sk - w.Sq) + 1) if w.causal else np.full(rows.shape, w.Sk)
        return float(4.0 * w.d * np.maximum(keys, 0).sum())

    rng = np.random.default_rng(seed + 12345)
    total_rows = w.B * w.Hq * w.Sq
    probe = rng.integers(0, total_rows, size=16, dtype=np.int64)
    t = time.perf_counter()
    oracle.attention_fwd_rows(q, k, v, scale, w.causal, probe)
    dt = max(time.perf_counter() - t, 1e-4)
    n = int(max(16, min(total_rows, 16 * seconds / dt)))
    rows = np.sort(rng.integers(0, total_rows, size=n, dtype=np.int64))
    t = time.perf_counter()
    oracle.attention_fwd_rows(q, k, v, scale, w.causal, rows)
    dt = time.perf_counter() - t
    f = flops_of(rows)
    return f / dt, f, oracle.num_threads(), f"{n} seeded random query rows of {total_rows}"


def oracle_bwd_rate(w: workloads.Workload, q, k, v, seed: int = 0) -> Tuple[float, int, str]:
    """Time the fp64 backward reference on one (batch, query head) of the
    workload -- the smallest piece it computes whole -- with a seeded dO;
    returns (flop/s credited at 2.5x the forward FLOPs of that head, threads,
    sample)."""
    import torch
    from oracle import attn_bwd as ob
    kv = w.Hq // w.Hkv
    q1 = q[:1, :, :1].contiguous()
    k1, v1 = k[:1, :, :1].contiguous(), v[:1, :, :1].contiguous()
    do1 = torch.randn(q1.shape, generator=torch.Generator().manual_seed(seed + 77)).to(torch.bfloat16)
    t = time.perf_counter()
    ob.attention_bwd(q1, k1, v1, do1, w.scale, w.causal)
    dt = time.perf_counter() - t
    f = BWD_FLOP_FACTOR * w.flops / (w.B * w.Hq)
    return f / dt, torch.get_num_threads(), f"one (batch, head) of {w.B * w.Hq} (kv group {kv})"


def run_reference(args, w: workloads.Workload) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import build as oracle_build
    oracle_build.build()
    q, k, v = workloads.make_inputs(w, seed=0)
    per_step_s = max(0.2, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rate(w, q, k, v, per_step_s, seed=1000 + i)
    flops = 0.0
    secs = 0.0
    threads = 1
    sample = ""
    for i in range(args.steps):
        rate, f, threads, sample = oracle_rate(w, q, k, v, per_step_s, seed=i)
        flops += f
        secs += f / rate
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), sample_per_step=sample),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {sample}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg
def run_ours(args, w: workloads.Workload) -> None:
    import torch

    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import attention_forward_fa4_gb300 as fa4
    fa4.load_library()

    w_rank, batch_offset = shard_workload(w, rank, world)
    bwd = args.pass_ == "bwd"
    fp8 = args.precision == "fp8"
    if fp8 and (bwd or args.num_splits or args.exp2_emulation or w.d != 128):
        raise SystemExit("--precision fp8 times the plain head-dim-128 forward only")
    if fp8:
        q_h, k_h, v_h, qs, ks, vs = workloads.make_inputs_fp8(w_rank, seed=0,
                                                              batch_offset=batch_offset)
    else:
        q_h, k_h, v_h = workloads.make_inputs(w_rank, seed=0, batch_offset=batch_offset)
    stream = torch.cuda.Stream(device=dev)
    q = q_h.to(dev)
    k = k_h.to(dev)
    v = v_h.to(dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    kw = dict(tau=args.tau, exp2_emulation=args.exp2_emulation)
    if args.num_splits:
        kw.update(num_splits=args.num_splits,
                  workspace=torch.empty(fa4.splitkv_workspace_bytes(w_rank.B, w.Hq, w.Sq, w.d,
                                                                    args.num_splits),
                                        dtype=torch.uint8, device=dev))

    if bwd:
        # the backward's inputs: the forward's outputs and a seeded dO
        fa4.fwd_into(q, k, v, o, lse, w.causal, w.scale, stream=stream)
        g = torch.Generator().manual_seed(7 + batch_offset)
        do_h = torch.randn(q_h.shape, generator=g).to(torch.bfloat16)
        dout = do_h.to(dev)
        o_h, lse_h = o.cpu(), lse.cpu()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsb = torch.empty(fa4.bwd_workspace_bytes(w_rank.B, w.Hq, w.Sq, w.d), dtype=torch.uint8,
                          device=dev)

    # Buffer set 0 serves the device-timed region; the end-to-end run
    # alternates between set 0 and a second set on its own stream.
    sets = [dict(q=q, k=k, v=v, o=o, lse=lse, kw=kw)]
    if bwd:
        sets[0].update(dout=dout, dq=dq, dk=dk, dv=dv, wsb=wsb)

    def launch(b=0, st=None):
        S = sets[b]
        st = stream if st is None else st
        if bwd:
            fa4.bwd_into(S["q"], S["k"], S["v"], S["o"], S["dout"], S["lse"], S["dq"], S["dk"],
                         S["dv"], w.causal, w.scale, deterministic=args.deterministic,
                         workspace=S["wsb"], stream=st)
        elif fp8:
            fa4.fwd_fp8_into(S["q"], S["k"], S["v"], S["o"], S["lse"], qs, ks, vs, w.causal,
                             w.scale, tau=args.tau, stream=st)
        else:
            fa4.fwd_into(S["q"], S["k"], S["v"], S["o"], S["lse"], w.causal, w.scale, stream=st,
                         **S["kw"])

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            launch()
    torch.cuda.synchronize()
    code, detail = fa4.device_status(clear=True)
    if code != fa4.FA4_OK:
        raise SystemExit(f"kernel status {fa4.status_string(code)} {detail}")

    # ---- device-timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if not args.no_clocks else None
    time.sleep(0.3 if sampler else 0.0)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()                       # evict q/k/v/o from L2 between launches
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    kernel_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    code, detail = fa4.device_status(clear=True)
    if code != fa4.FA4_OK:
        raise SystemExit(f"kernel status {fa4.status_string(code)} {detail}")

    # ---- end to end: pinned host inputs in, host outputs out, every step
    q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    o_p = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    lse_p = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    if bwd:
        o_bp, lse_bp, do_p = o_h.pin_memory(), lse_h.pin_memory(), do_h.pin_memory()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    host_api = not bwd and not fp8 and not args.num_splits
    # Two streams, each with its own device buffers and host outputs, so one
    # step's copies overlap the other step's kernels.
    streams = [stream, torch.cuda.Stream(device=dev)]
    o_pp = [o_p, torch.empty(o.shape, dtype=o.dtype, pin_memory=True)]
    lse_pp = [lse_p, torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)]
    if host_api:
        # the plain forward through fa4_fwd_host: pinned host q, k, v in,
        # o, lse out, every step
        ws_e2e = [torch.empty(fa4.host_workspace_bytes(w_rank.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d),
                              dtype=torch.uint8, device=dev) for _ in range(2)]
    else:
        # torch copies from pinned host buffers around the device call
        S1 = {n: torch.empty_like(t) for n, t in sets[0].items() if isinstance(t, torch.Tensor)}
        S1["kw"] = dict(kw)
        if "workspace" in kw:
            S1["kw"]["workspace"] = torch.empty_like(kw["workspace"])
        sets.append(S1)
        if bwd:
            grads_pp = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
                        for _ in range(2)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    if host_api:
        main = torch.cuda.current_stream(dev)
        e_start.record(main)
        for st in streams:
            st.wait_event(e_start)
        for i in range(e2e_steps):
            fa4.fwd_host_into(q_p, k_p, v_p, o_pp[i % 2], lse_pp[i % 2], w.causal, w.scale,
                              workspace=ws_e2e[i % 2], tau=args.tau,
                              exp2_emulation=args.exp2_emulation, stream=streams[i % 2])
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            main.wait_event(ev)
        e_end.record(main)
    else:
        main = torch.cuda.current_stream(dev)
        e_start.record(main)
        for st in streams:
            st.wait_event(e_start)
        for i in range(e2e_steps):
            b = i % 2
            S = sets[b]
            with torch.cuda.stream(streams[b]):
                S["q"].copy_(q_p, non_blocking=True)
                S["k"].copy_(k_p, non_blocking=True)
                S["v"].copy_(v_p, non_blocking=True)
                if bwd:
                    S["o"].copy_(o_bp, non_blocking=True)
                    S["lse"].copy_(lse_bp, non_blocking=True)
                    S["dout"].copy_(do_p, non_blocking=True)
                launch(b, streams[b])
                if bwd:
                    for dst, src in zip(grads_pp[b], (S["dq"], S["dk"], S["dv"])):
                        dst.copy_(src, non_blocking=True)
                else:
                    o_pp[b].copy_(S["o"], non_blocking=True)
                    lse_pp[b].copy_(S["lse"], non_blocking=True)
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            main.wait_event(ev)
        e_end.record(main)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_end)
    code, detail = fa4.device_status(clear=True)
    if code != fa4.FA4_OK:
        raise SystemExit(f"kernel status {fa4.status_string(code)} {detail}")
    last = (e2e_steps - 1) % 2
    if bwd:   # dK, dV are accumulated in one CTA each: bit-identical run to run
        same = all(torch.equal(hp, t.cpu()) for hp, t in zip(grads_pp[last][1:], (dk, dv)))
    else:
        same = torch.equal(o_pp[last], o.cpu()) and torch.equal(lse_pp[last], lse.cpu())
    if not same:
        raise SystemExit("end-to-end output differs from the device-resident run")
    h2d = (q.numel() + k.numel() + v.numel()) * q.element_size()
    d2h = o.numel() * 2 + lse.numel() * 4

    # ---- copy roofline of the end-to-end step: the same host<->device copies
    # (one per tensor, same pinned buffers, two alternating streams) with no
    # kernel in between
    ins_h = [q_p, k_p, v_p] + ([o_bp, lse_bp, do_p] if bwd else [])
    outs_h = [grads_pp[b] for b in range(2)] if bwd else [[o_pp[b], lse_pp[b]] for b in range(2)]
    outs_src = [dq, dk, dv] if bwd else [o, lse]
    ins_dev = [[torch.empty(t.shape, dtype=t.dtype, device=dev) for t in ins_h] for _ in range(2)]
    outs_dev = [[torch.empty_like(t) for t in outs_src] for _ in range(2)]
    torch.cuda.synchronize()
    c_start = torch.cuda.Event(enable_timing=True)
    c_end = torch.cuda.Event(enable_timing=True)
    main = torch.cuda.current_stream(dev)
    c_start.record(main)
    for st in streams:
        st.wait_event(c_start)
    for i in range(e2e_steps):
        b = i % 2
        with torch.cuda.stream(streams[b]):
            for dst, src in zip(ins_dev[b], ins_h):
                dst.copy_(src, non_blocking=True)
            for dst, src in zip(outs_h[b], outs_dev[b]):
                dst.copy_(src, non_blocking=True)
    for st in streams:
        ev = torch.cuda.Event()
        ev.record(st)
        main.wait_event(ev)
    c_end.record(main)
    torch.cuda.synchronize()
    copy_ms = c_start.elapsed_time(c_end)
    del ins_dev, outs_dev

    if bwd:
        h2d += o.numel() * 2 + lse.numel() * 4 + dout.numel() * 2
        d2h = (dq.numel() + dk.numel() + dv.numel()) * 2

    if pg:
        kernel_ms, e2e_ms = max_over_ranks([kernel_ms, e2e_ms], pg, dev)

    flops_rank_step = w_rank.flops * (BWD_FLOP_FACTOR if bwd else 1.0)
    value = flops_rank_step * args.steps * world / (kernel_ms * 1e-3) / 1e12
    e2e_value = flops_rank_step * e2e_steps * world / (e2e_ms * 1e-3) / 1e12
    per_launch_ms = kernel_ms / args.steps
    achieved = flops_rank_step / (per_launch_ms * 1e-3) / 1e12
    peaks = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_source = f"{peaks['_source']} bf16_tflops (burst)"
    if fp8:
        fp8_peak = fp8_gemm_peak_tflops(dev) if rank == 0 else None
        if fp8_peak:
            peak = fp8_peak
            peak_source = "measured here: e4m3 GEMM 8192^3 (torch._scaled_mm), best of 10"
        else:
            peak *= FP8_OVER_BF16
            peak_source += f" x {FP8_OVER_BF16:g} (nominal FP8:BF16 dense ratio)"

    # lazy-rescale counts of this workload: 32-row-group steps (after each
    # tile's first key block) that rescaled the output, at tau and at 0
    rescale = None
    if not bwd and not args.no_rescale_stats:
        cnt = {}
        for tau in (args.tau, 0.0):
            stats = torch.zeros(2, dtype=torch.int64, device=dev)
            if fp8:
                fa4.fwd_fp8_into(q, k, v, o, lse, qs, ks, vs, w.causal, w.scale, tau=tau,
                                 rescale_stats=stats, stream=stream)
            else:
                fa4.fwd_into(q, k, v, o, lse, w.causal, w.scale, tau=tau, rescale_stats=stats,
                             stream=stream, **{k_: v_ for k_, v_ in kw.items() if k_ != "tau"})
            torch.cuda.synchronize()
            cnt[tau] = stats.cpu().tolist()
        r_tau, steps = cnt[args.tau]
        r_eager = cnt[0.0][0]
        rescale = {"tau": args.tau, "row_group_steps": steps, "rescales": r_tau,
                   "rescales_at_tau_0": r_eager,
                   "fewer_by": (r_eager / r_tau) if r_tau else None}
    traffic = (stored_traffic(w.name, "fa4_bwd_kernel") if bwd else
               stored_traffic(w.name + ("_fp8" if fp8 else "")
                              + (f"_split{args.num_splits}" if args.num_splits else "")))

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline and bwd:
            rate, threads, sample = oracle_bwd_rate(w, q_h, k_h, v_h)
            cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": sample}
        elif world == 1 and not args.no_cpu_baseline and fp8:
            # the FP8 oracle's forward equals the fp64 definition on the e4m3
            # values (exact in BF16) with the scales folded into scale and O
            from oracle import fp8 as o8
            deq = [torch.from_numpy(o8.e4m3_to_float(o8.codes_of(t))).to(torch.bfloat16)
                   for t in (q_h, k_h, v_h)]
            rate, _, threads, sample = oracle_rate(w, *deq, args.cpu_seconds,
                                                   scale=w.scale * qs * ks)
            cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": sample + " (fp64 definition on the dequantised e4m3 inputs)"}
        elif world == 1 and not args.no_cpu_baseline:
            rate, _, threads, sample = oracle_rate(w, q_h, k_h, v_h, args.cpu_seconds)
            cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": sample}
        line = {
            "metric": METRIC_BWD if bwd else (METRIC_FP8 if fp8 else METRIC), "value": value,
            "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_launch_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if fp8 else "bf16",
            "data": "synthetic",
            "config": dict(w.describe(), global_batch=w.B * world, parallelism=f"replica-shards{world}",
                           **({"dtype_in": "e4m3 (per-tensor scales amax/448)"} if fp8 else {}),
                           l2="flushed before every timed launch (256 MiB write)",
                           tau=args.tau, exp2_emulation=args.exp2_emulation,
                           num_splits=args.num_splits, precision=args.precision,
                           **{"pass": args.pass_},
                           **({"deterministic": args.deterministic} if bwd else {})),
            "pct_of_2250_tflops": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
            **({"pct_of_4500_tflops": 100.0 * value / world / (2 * NOMINAL_BF16_TFLOPS)}
               if fp8 else {}),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": peak_source,
                         "traffic": traffic["bytes"] if traffic else None,
                         "traffic_source": traffic["source"] if traffic else None,
                         "algorithmic_bytes": (w_rank.hbm_bytes_bwd if bwd else
                                               w_rank.hbm_bytes_fp8 if fp8 else w_rank.hbm_bytes)},
            "cpu_baseline": cpu,
            "clocks": clocks,
            "rescale_stats": rescale,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "copy_roofline": {
                        "what": ("the step's host<->device copies alone: same tensors, pinned "
                                 "buffers and two alternating streams, no kernel"),
                        "bytes_per_step": h2d + d2h,
                        "ms_per_step": copy_ms / e2e_steps,
                        "gbs": (h2d + d2h) * e2e_steps / (copy_ms * 1e-3) / 1e9,
                        "e2e_ms_per_step": e2e_ms / e2e_steps,
                        "frac": copy_ms / e2e_ms},
                    "api": ("fa4_fwd_host (pinned host buffers, copies inside the call), "
                            "2 streams alternating" if host_api else
                            "torch copies from pinned host buffers around the call, "
                            "2 streams alternating")},
            "gpu_launches": args.steps * (3 if bwd else (2 if args.num_splits else 1)),
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def main(argv: Optional[List[str]] = None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.LONG_CAUSAL.name,
                    choices=[x.name for x in workloads.ALL_NAMED + workloads.EXTRA])
    ap.add_argument("--tau", type=float, default=8.0)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward (dQ, dK, dV)")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="key-range split forward with this many splits (0: plain forward)")
    ap.add_argument("--exp2-emulation", type=int, choices=[0, 4, 8], default=0,
                    help="one softmax entry pair in N through the software 2^x (0: none)")
    ap.add_argument("--precision", choices=["bf16", "fp8"], default="bf16",
                    help="fp8: e4m3 Q, K, V (per-tensor scales) through fa4_fwd_fp8")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward only: dQ tiles added in key-block order (fa4_bwd_ex)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-rescale-stats", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = workloads.by_name(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
