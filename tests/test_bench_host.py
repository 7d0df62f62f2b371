"""Host-side logic of the benchmark: the closed-form roofline of
"FlashAttention-4" Table 1, the weak-scaling shard plan and the
max-over-ranks timing reduction on a two-rank gloo group."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads
from tests import golden


def test_table1_roofline_cycles_at_b200_constants():
    # The pages' printed cycle counts (tests/golden, with the citation).
    t = golden.load("table1_forward_roofline_b200.txt")
    c = bench.table1_cycles(int(t["M"]), int(t["N"]), int(t["d"]), flops_per_clk=t["flops_per_clk"],
                            exp_per_clk=t["exp_per_clk"], smem_bytes_per_clk=t["smem_bytes_per_clk"])
    assert c == {"mma": t["mma"], "exp": t["exp"], "smem": t["smem"]}
    # GB300 doubles MUFU throughput: exp halves, MMA and SMEM unchanged.
    g = bench.table1_cycles(256, 128, 128, exp_per_clk=32.0)
    assert g["exp"] == 1024.0 and g["mma"] == 2048.0
    # d = 64: MMA and SMEM halve, exp does not -> exp-bound regime.
    h = bench.table1_cycles(256, 128, 64, exp_per_clk=32.0)
    assert h["mma"] == 1024.0 and h["exp"] == 1024.0 and h["smem"] == 768.0


def test_workload_flops_and_bytes():
    w = workloads.LONG_CAUSAL
    assert w.flops == 4 * 2 * 16 * 8192 * 8192 * 128 / 2
    assert w.hbm_bytes == 4 * (2 * 8192 * 16 * 128 * 2) + 2 * 16 * 8192 * 4
    g = workloads.GQA_STRESS
    assert g.hbm_bytes == 2 * (16384 * 32 * 128 * 2) + 2 * (16384 * 8 * 128 * 2) + 32 * 16384 * 4


def test_shards_are_disjoint_and_cover_the_global_batch():
    w = workloads.MID
    seen = []
    for r in range(4):
        wr, off = bench.shard_workload(w, r, 4)
        assert wr.B == w.B
        seen.extend(range(off, off + wr.B))
    assert sorted(seen) == list(range(4 * w.B))
    with pytest.raises(ValueError):
        bench.shard_workload(w, 4, 4)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.Workload("t", 1, 2, 2, 16, 16, 8, False)
        wr, off = bench.shard_workload(w, rank, world)
        q, _, _ = workloads.make_inputs(wr, seed=0, batch_offset=off)
        # each rank reports a different "time"; the job time is the max
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
        digest = float(q.float().sum())
        out.put((rank, got, digest))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_over_ranks_and_distinct_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == [2.0, 10.0]
    assert res[0][2] != res[1][2]          # ranks drew different data
