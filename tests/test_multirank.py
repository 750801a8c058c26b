"""The benchmark's N-rank path on CPU ranks (gloo, world size 2): every rank
works on its own batch (no collective on the data path); the only collective
is the max over ranks of the timings, and the job rate counts every rank's
units over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import dsa_workloads as W
    # each rank draws its own batch from a rank-specific seed
    spec = W.SPECS["tiny"].scaled(seed=W.SPECS["tiny"].seed + 100 * rank)
    wl = W.make_workload(spec)
    local_ms = [10.0 + 5.0 * rank, 3.0 - rank]
    mx = bench.max_over_ranks(local_ms, torch.device("cpu"))
    out[rank] = (mx, bench.job_throughput(wl.total_q, world, 7, mx[0]), float(wl.k_idx.float().sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_cpu_ranks_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (mx0, v0, s0), (mx1, v1, s1) = out[0], out[1]
    assert mx0 == mx1 == [15.0, 3.0]                       # max over ranks, seen by all ranks
    assert v0 == pytest.approx(16 * 2 * 7 / 0.015)         # 16 queries per rank, 2 ranks, 7 steps
    assert s0 != s1                                        # independent batches per rank
