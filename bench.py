"""Benchmark of the DSA forward path (indexer + top-k + sparse MLA, k = 2048).

One step = one dsa_forward call over the decode workload: 32 sequences x
context 32768, one query token each; indexer 64 heads x 128 dims; top-k 2048;
sparse MLA in MQA mode with 64 heads over a 576-dim latent (values 512).
Metric: query tokens/s, whole job (all ranks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the float64 CPU oracle (the only reference this
project has) on a bounded sample of the same workload.
Under torchrun each rank runs its own 32-sequence batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

if "OPENBLAS_NUM_THREADS" not in os.environ:  # the oracle's BLAS: every host core, stated in the line
    os.environ["OPENBLAS_NUM_THREADS"] = str(os.cpu_count() or 1)

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dsa_workloads as W  # noqa: E402

METRIC = "DSA query tokens/s (indexer+top-k+sparse MLA) at k=2048; % HBM roofline"
WORKLOAD = "decode"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _config(spec):
    return {"workload": f"{spec.name}: B={spec.batch} x ctx {spec.ctx_len}, {spec.q_per_seq} query/seq; "
                        f"indexer {spec.idx_heads}x{spec.idx_dim}; top-k {spec.topk}; MQA {spec.heads} heads, "
                        f"latent {spec.d_qk} (value {spec.d_v})",
            "global_batch": spec.batch * spec.q_per_seq, "seq_len": spec.ctx_len, "topk": spec.topk}


def _shape(wl):
    from long_context_lightning_gb300 import accounting
    s = wl.spec
    seq, pos = wl.query_positions()
    return accounting.Shape(n=[p + 1 for p in pos], seq_of=seq, idx_heads=s.idx_heads, idx_dim=s.idx_dim,
                            topk=s.topk, heads=s.heads, d_qk=s.d_qk, d_v=s.d_v, n_layers=s.n_layers)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.gpu = None
        try:  # nvidia-smi ignores CUDA_VISIBLE_DEVICES: address the GPU by its UUID
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.gpu = vis.split(",")[device.index or 0] if vis else str(device.index or 0)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_baseline(spec, wl_cpu, budget_s=12.0):
    """The oracle, as it stands, on the host cores: whole decode queries until the budget is spent."""
    import oracle
    t0 = time.perf_counter()
    done = 0
    T = wl_cpu.total_q
    while True:
        oracle.dsa_forward(wl_cpu, queries=[done % T])
        done += 1
        if time.perf_counter() - t0 > budget_s or done >= 4 * T:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "query tokens/s", "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle",
            "sample": f"{done} decode queries (each: indexer over 32768 keys, top-{spec.topk}, 64-head MLA over "
                      f"{spec.topk} rows) of the {spec.batch}-query batch, float64 numpy, {dt:.1f} s"}


def run_reference(args, rank, world):
    spec = W.SPECS[WORKLOAD]
    if rank != 0:
        return
    import oracle
    wl = W.make_workload(spec, device="cuda" if torch.cuda.is_available() else "cpu").to("cpu")
    T = wl.total_q
    per_step = 2                                   # queries per reference step (bounded sample)
    q = 0
    for _ in range(args.warmup):
        oracle.dsa_forward(wl, queries=[(q + i) % T for i in range(per_step)])
        q += per_step
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.dsa_forward(wl, queries=[(q + i) % T for i in range(per_step)])
        q += per_step
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    cores = int(os.environ["OPENBLAS_NUM_THREADS"])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(spec),
            "cpu_baseline": {"value": value, "unit": "query tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} decode queries per step (float64 numpy oracle)"},
            "e2e": {"value": value, "unit": "query tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings (every rank gets the result)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized() and \
            torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(units_per_rank: int, world: int, steps: int, max_total_ms: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world * steps / (max_total_ms / 1e3)


def _traffic_from_profile(kernel_file: str, summary: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "long_context_lightning_gb300", "csrc", kernel_file)
    try:
        with open(src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        with open(path) as f:
            txt = f.read()
        vals = {}
        for line in txt.splitlines():
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") != h:
            return None
        return float(vals["dram_bytes_per_launch"])
    except Exception:
        return None


def run_gpu(args, rank, world, local_rank):
    import __graft_entry__
    from long_context_lightning_gb300 import _lib
    from long_context_lightning_gb300 import accounting
    from long_context_lightning_gb300.api import SparseAttention

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    _lib.load()
    spec = W.SPECS[WORKLOAD].scaled(seed=W.SPECS[WORKLOAD].seed + 100 * rank)
    wl = W.make_workload(spec, device=dev)
    sa = SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, spec.d_v,
                         spec.scale, spec.topk, seq_start=wl.seq_start)
    stream = torch.cuda.current_stream(dev)
    sa.forward()
    torch.cuda.synchronize(dev)
    status = _lib.check_device_error()
    if status != _lib.DSA_OK:
        raise RuntimeError(f"device error after the first forward: {_lib.status_string(status)}")

    # one forward captured in a CUDA graph (4 launches: plan, indexer, top-k, sparse MLA)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        sa.forward()
    torch.cuda.synchronize(dev)
    launches_per_step = 4

    # L2 flush between timed steps: write 512 MB (> the 129 MB L2), then read a
    # 256 MB buffer so the lines left in L2 are clean (no write-back lands in
    # the next timed step)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    scrub = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def flush_l2(i):
        flush.fill_(i)
        scrub.sum()
    clocks = ClockSampler(dev)
    clocks.start()
    # warm-up: W graph replays, then enough extra replays for the clocks to settle under load
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    t_busy = time.perf_counter()
    while time.perf_counter() - t_busy < 0.5:
        for _ in range(50):
            graph.replay()
        torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i)                         # between timed steps, outside the events
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)

    # per-kernel times on the same stream (marks between the launches), same flushing
    n_brk = min(args.steps, 200)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_brk)]
    for row in marks:          # torch creates the CUDA event on first record
        for m in row:
            m.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(n_brk):
        flush_l2(i)
        _lib.forward_marked(sa.batch, sa.indexer, sa.topk, sa.layers, sa.idx, sa.outs, sa.lses, sa.workspace,
                            marks[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per = {"plan": [], "indexer": [], "topk": [], "sparse_mla": []}
    for m in marks:
        for j, name in enumerate(per):
            per[name].append(m[j].elapsed_time(m[j + 1]))
    kern_ms = {k: statistics.mean(v) for k, v in per.items()}

    # end to end through the public API: inputs from pinned host memory, results back
    host_in = [t.cpu().pin_memory() for t in
               (wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.seq_start, *wl.q, *wl.kv)]
    dev_in = [wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.seq_start, *wl.q, *wl.kv]
    host_out = [sa.idx.cpu().pin_memory()] + [o.cpu().pin_memory() for o in sa.outs] + \
               [x.cpu().pin_memory() for x in sa.lses]
    dev_out = [sa.idx] + list(sa.outs) + list(sa.lses)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    n_e2e = max(3, min(args.steps, 20))
    for _ in range(2):
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        sa.forward()
        for h, d in zip(host_out, dev_out):
            h.copy_(d, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        sa.forward()
        for h, d in zip(host_out, dev_out):
            h.copy_(d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    status = _lib.check_device_error()
    if status != _lib.DSA_OK:
        raise RuntimeError(f"device error during the benchmark: {_lib.status_string(status)}")

    # aggregate over ranks: max time
    T = wl.total_q
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dev)
    if rank != 0:
        return
    value = job_throughput(T, world, args.steps, total_ms)
    hbm, tf, peak_kind = _peaks()
    shp = _shape(wl)
    idx_bytes = accounting.indexer_bytes(shp)
    mla_bytes = accounting.mla_bytes(shp)
    all_bytes = accounting.forward_bytes(shp)
    idx_gbs = idx_bytes / (kern_ms["indexer"] * 1e-3) / 1e9
    mla_gbs = mla_bytes / (kern_ms["sparse_mla"] * 1e-3) / 1e9
    traffic = _traffic_from_profile("indexer.cu", "indexer_decode_b32_ctx32k.md")
    wl_cpu = wl.to("cpu")
    cpu = _cpu_baseline(spec, wl_cpu) if world == 1 or rank == 0 else None
    line = {
        "metric": METRIC, "value": value, "unit": "query tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**_config(spec), "parallelism": f"dp{world} (independent batches per GPU)",
                   "l2": "flushed between timed steps (512 MB write + 256 MB read, outside the timed events)",
                   "cuda_graph": True},
        "roofline": {"bound": "hbm", "kernel": "indexer", "achieved": idx_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": idx_gbs / hbm, "traffic": traffic, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": idx_bytes},
        "kernels_ms": kern_ms,
        "sparse_mla_roofline": {"bound": "hbm", "achieved": mla_gbs, "peak": hbm, "unit": "GB/s",
                                "frac": mla_gbs / hbm, "algorithmic_bytes_per_launch": mla_bytes},
        "step_roofline": {"bound": "hbm", "achieved": all_bytes / (total_ms / args.steps * 1e-3) / 1e9,
                          "peak": hbm, "unit": "GB/s",
                          "frac": all_bytes / (total_ms / args.steps * 1e-3) / 1e9 / hbm,
                          "algorithmic_bytes_per_step": all_bytes},
        "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "query tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "native" else "gloo"
        if args.impl == "native":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
