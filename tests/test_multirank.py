"""The benchmark's N-rank path on CPU ranks (gloo, world size 2).

Every rank works on its own seeded batch (no collective on the data path):
here each rank runs the float64 oracle over its own tiny batch, times that
work, and the ranks agree on the slowest rank's time with the benchmark's own
max_over_ranks; the job rate then counts every rank's query tokens over that
time (job_throughput).  The test checks the aggregation against the per-rank
timings the ranks actually measured, and that the ranks' work differed.
"""
import os
import socket
import time

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
    import numpy as np

    import bench
    import dsa_workloads as W
    import oracle
    # each rank draws its own batch from a rank-specific seed, as bench.py does
    spec = W.SPECS["tiny"].scaled(seed=W.SPECS["tiny"].seed + 100 * rank)
    wl = W.make_workload(spec)
    steps = 2
    t0 = time.perf_counter()
    for _ in range(steps):
        res = oracle.dsa_forward(wl)
    local_ms = (time.perf_counter() - t0) * 1e3
    # the work is real: every query selected k positions inside its causal context
    seq, pos = wl.query_positions()
    for t in range(wl.total_q):
        assert len(res.idx[t]) == spec.topk and res.idx[t].max() <= pos[t]
    digest = float(sum(float(np.abs(res.out[0][t]).sum()) for t in range(wl.total_q)))
    mx = bench.max_over_ranks([local_ms], torch.device("cpu"))
    rate = bench.job_throughput(wl.total_q, world, steps, mx[0])
    out[rank] = (local_ms, mx[0], rate, wl.total_q, steps, digest)
    dist.barrier()
    dist.destroy_process_group()


def test_two_cpu_ranks_run_their_own_batches_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")  # no fork of this (threaded) test process, the manager's included
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    (ms0, mx0, rate0, T0, steps, d0), (ms1, mx1, rate1, T1, _, d1) = out[0], out[1]
    # every rank sees the slowest rank's measured time
    assert mx0 == mx1 == pytest.approx(max(ms0, ms1))
    # whole-job rate: all ranks' query tokens over the slowest rank's time
    assert rate0 == rate1 == pytest.approx((T0 + T1) * steps / (max(ms0, ms1) / 1e3))
    # independent batches per rank: different inputs, different attention outputs
    assert d0 != d1
