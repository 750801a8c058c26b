"""Benchmark of the DSA forward path (indexer + top-k + sparse MLA, k = 2048).

One step = one dsa_forward call over the decode workload: 32 sequences x
context 32768, one query token each; indexer 64 heads x 128 dims; top-k 2048;
sparse MLA in MQA mode with 64 heads over a 576-dim latent (values 512).
Metric: query tokens/s, whole job (all ranks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the float64 CPU oracle (the only reference this
project has) on a bounded sample of the same workload.  `e2e` is a decode step
as a server runs it: the step's queries and the new tokens' cache rows copied
from pinned host memory, appended into the resident caches, the forward, and
the results copied back.
Under torchrun each rank runs its own 32-sequence batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line.

Beside the decode headline, the line carries `per_config`: the tiny,
chunked-prefill, ragged-paged and IndexShare workloads and two compressed-entry
workloads (top-512 and top-1024 of one entry per 4 tokens), each timed the same
way (CUDA-graph replay of the fused call, CUDA events on the launching stream,
L2 flushed between steps) with its dominant kernel's roofline and the oracle
timed on a bounded sample beside it.  For IndexShare one query token is one
query through the whole 4-layer group.  `per_config.hisparse` times the HBM
row cache over pinned host memory on the decode workload (cold, warm and
decode-like steps) and sparse MLA over its slots.  `per_config.mha` times MHA mode
(per-head up-projection of a 4608-token context and attention of 64 heads
over each query's selection) on its prefill-chunk workload.
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


def _config(spec):
    return {"workload": f"{spec.name}: B={spec.batch} x ctx {spec.ctx_len}, {spec.q_per_seq} query/seq; "
                        f"indexer {spec.idx_heads}x{spec.idx_dim}; top-k {spec.topk}; MQA {spec.heads} heads, "
                        f"latent {spec.d_qk} (value {spec.d_v})",
            "global_batch": spec.batch * spec.q_per_seq, "seq_len": spec.ctx_len, "topk": spec.topk}


def _shape(wl):
    from long_context_lightning_gb300 import accounting
    s = wl.spec
    seq, pos = wl.query_positions()
    # causal context in cache entries (tokens, or complete blocks of compress_ratio tokens)
    return accounting.Shape(n=[(p + 1) // s.compress_ratio for p in pos], seq_of=seq, idx_heads=s.idx_heads,
                            idx_dim=s.idx_dim,
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


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# kernel from one ncu capture, keyed by workload and kernel, with the first 16
# hex digits of the sha256 of the kernel's source file when it was captured.
# A source that has changed since makes the figure stale: it is reported as
# null.  Captured with
#   ncu --set full --clock-control none -k regex:<kernel>_kernel -s <n> -c <1..3> \
#       -o <report> python bench.py --steps 5 --warmup 3 --no-per-config
# (the exact command of each capture is kept with its ncu summary)
NCU_TRAFFIC = {
    ("decode", "indexer"): ("indexer.cu", "5f358bf61f8aaa44", 273867264.0),
    ("decode", "topk"): ("topk.cu", "51834c3a49681375", 4273664.0),
    ("decode", "sparse_mla"): ("sparse_mla.cu", "c4a76ec2f68182a4", 82548736.0),
}


def _traffic(workload: str, kernel: str):
    entry = NCU_TRAFFIC.get((workload, kernel))
    if entry is None:
        return None
    src, sha, nbytes = entry
    try:
        with open(os.path.join(ROOT, "long_context_lightning_gb300", "csrc", src), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return nbytes if h == sha else None


def _peaks_all():
    """HBM copy GB/s, bf16 TFLOP/s burst and sustained, and where they come from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


KERNELS = ("plan", "indexer", "topk", "sparse_mla")


def _staging(parts, dev):
    """One pinned host buffer and one device buffer holding `parts` (each piece
    256-byte aligned), the host copy filled from `parts`; returns both buffers
    and the pieces' views in each."""
    offs, n = [], 0
    for t in parts:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    devb = torch.empty(n, dtype=torch.uint8, device=dev)
    hv, dv = [], []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        hv.append(host[o:o + nb].view(t.dtype).view(t.shape))
        dv.append(devb[o:o + nb].view(t.dtype).view(t.shape))
        hv[-1].copy_(t.cpu())
    return host, devb, hv, dv


class _Run:
    """One workload resident on the device, its fused call captured in a CUDA graph."""

    def __init__(self, spec, dev):
        from long_context_lightning_gb300 import _lib
        from long_context_lightning_gb300.api import SparseAttention
        self.spec = spec
        self.dev = dev
        self.wl = W.make_workload(spec, device=dev)
        wl = self.wl
        self.sa = SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, spec.d_v,
                                  spec.scale, spec.topk, seq_start=wl.seq_start, page_table=wl.page_table,
                                  page_size=spec.page_size, compress_ratio=spec.compress_ratio)
        self.sa.forward()
        torch.cuda.synchronize(dev)
        status = _lib.check_device_error()
        if status != _lib.DSA_OK:
            raise RuntimeError(f"{spec.name}: device error after the first forward: {_lib.status_string(status)}")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            self.sa.forward()
        torch.cuda.synchronize(dev)

    def time_steps(self, steps, warmup, flush_l2, stream, settle_s=0.0):
        """CUDA-event time of each of `steps` graph replays, L2 flushed before each (outside the events)."""
        for _ in range(max(warmup, 3)):
            self.graph.replay()
        t_busy = time.perf_counter()
        while time.perf_counter() - t_busy < settle_s:
            for _ in range(50):
                self.graph.replay()
            torch.cuda.synchronize(self.dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize(self.dev)
        for i in range(steps):
            flush_l2(i)
            starts[i].record(stream)
            self.graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]

    def kernel_ms(self, n, flush_l2, stream):
        """Mean time of each launch from a separate run of dsa_forward_marked (events between the launches;
        the marks stop programmatic overlap, so the means add up to more than a step)."""
        from long_context_lightning_gb300 import _lib
        sa = self.sa
        marks = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
        for row in marks:          # torch creates the CUDA event on first record
            for m in row:
                m.record(stream)
        torch.cuda.synchronize(self.dev)
        for i in range(n):
            flush_l2(i)
            _lib.forward_marked(sa.batch, sa.indexer, sa.topk, sa.layers, sa.idx, sa.outs, sa.lses, sa.workspace,
                                marks[i], compress_ratio=self.spec.compress_ratio)
        torch.cuda.synchronize(self.dev)
        per = {k: [] for k in KERNELS}
        for m in marks:
            for j, name in enumerate(KERNELS):
                per[name].append(m[j].elapsed_time(m[j + 1]))
        return {k: statistics.mean(v) for k, v in per.items()}

    def check(self, what):
        from long_context_lightning_gb300 import _lib
        status = _lib.check_device_error()
        if status != _lib.DSA_OK:
            raise RuntimeError(f"{what}: device error: {_lib.status_string(status)}")


# nominal GB300 figures, reported beside the measured-peak fractions: HBM3e
# bandwidth (about 8 TB/s) and the dense bf16 tensor rate
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def _with_nominal(roof):
    nominal = NOMINAL_HBM_GBS if roof["unit"] == "GB/s" else NOMINAL_BF16_TFLOPS
    roof["nominal_peak"] = nominal
    roof["frac_of_nominal"] = roof["achieved"] / nominal
    return roof


def _roofline(wl, kern_ms, peaks, workload):
    """Dominant kernel's roofline (HBM bytes or tensor FLOPs, algorithmic), plus the sparse MLA's and the
    whole step's byte fractions."""
    from long_context_lightning_gb300 import accounting as A
    hbm, tf_burst, tf_sust, kind = peaks
    shp = _shape(wl)
    work = {
        "indexer": (A.indexer_bytes(shp), A.indexer_flops(shp)),
        "topk": (A.topk_bytes(shp), 0),
        "sparse_mla": (A.mla_bytes(shp), A.mla_flops(shp)),
    }
    dom = max(("indexer", "topk", "sparse_mla"), key=lambda k: kern_ms[k])
    nbytes, flops = work[dom]
    sec = kern_ms[dom] * 1e-3
    # a kernel whose FLOPs per byte exceed the ridge of the measured peaks is tensor-bound
    ridge = tf_sust * 1e12 / (hbm * 1e9)
    if flops and flops / max(nbytes, 1) > ridge:
        ach = flops / sec / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tf_sust, "unit": "TFLOP/s",
                "frac": ach / tf_sust, "traffic": _traffic(workload, dom), "peak_kind": f"{kind} (bf16 sustained)",
                "algorithmic_flops_per_launch": flops}
    else:
        ach = nbytes / sec / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": _traffic(workload, dom), "peak_kind": kind, "algorithmic_bytes_per_launch": nbytes}
    mla_b, mla_f = work["sparse_mla"]
    mla_gbs = mla_b / (kern_ms["sparse_mla"] * 1e-3) / 1e9
    mla = {"bound": "hbm", "achieved": mla_gbs, "peak": hbm, "unit": "GB/s", "frac": mla_gbs / hbm,
           "traffic": _traffic(workload, "sparse_mla"), "algorithmic_bytes_per_launch": mla_b,
           "tflops": mla_f / (kern_ms["sparse_mla"] * 1e-3) / 1e12}
    return _with_nominal(roof), _with_nominal(mla), A.forward_bytes(shp), A.forward_flops(shp)


def _oracle_sample(wl, queries, kv_on_device=False, min_s=2.0):
    """The oracle as it stands, query by query over `queries` (cycled) until at least `min_s` seconds of
    work are done; (seconds, queries done)."""
    import oracle
    fetch = None
    if kv_on_device:
        fetch = lambda layer, rows: wl.kv[layer][torch.from_numpy(rows).to(wl.kv[layer].device)].cpu()  # noqa: E731
        cpu = wl.to("cpu", kv_too=False)
    else:
        cpu = wl.to("cpu")
    t0 = time.perf_counter()
    done = 0
    while True:
        oracle.dsa_forward(cpu, queries=[queries[done % len(queries)]], kv_rows_fetch=fetch)
        done += 1
        if time.perf_counter() - t0 >= min_s and done >= min(len(queries), 4):
            break
    return time.perf_counter() - t0, done


# per workload: which queries the CPU baseline cycles through (about 2-4 s of work each)
CPU_SAMPLE = {
    "tiny": (lambda T: list(range(T)), "queries of the 16-query chunk, cycled"),
    "prefill": (lambda T: [0, T // 2, T - 1, 1, T // 4, 3 * T // 4], "chunk queries at 0, T/4, T/2, 3T/4, T-1 and 1"),
    "ragged": (lambda T: list(range(T)), "ragged queries in order"),
    "indexshare": (lambda T: list(range(T)), "queries through all 4 layers"),
    "csa_flash": (lambda T: list(range(T)), "decode queries over compressed entries, in order"),
    "csa_pro": (lambda T: list(range(T)), "decode queries over compressed entries, in order"),
}


def run_gpu(args, rank, world, local_rank):
    import __graft_entry__
    from long_context_lightning_gb300 import _lib

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    _lib.load()
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks_all()
    hbm = peaks[0]

    # L2 flush between timed steps: write 512 MB (> the 129 MB L2), then read a
    # 256 MB buffer so the lines left in L2 are clean (no write-back lands in
    # the next timed step)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    scrub = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def flush_l2(i):
        flush.fill_(i)
        scrub.sum()

    spec = W.SPECS[WORKLOAD].scaled(seed=W.SPECS[WORKLOAD].seed + 100 * rank)
    run = _Run(spec, dev)
    wl, sa = run.wl, run.sa
    launches_per_step = 4      # plan, indexer, top-k, sparse MLA

    clocks = ClockSampler(dev)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    step_ms = run.time_steps(args.steps, args.warmup, flush_l2, stream, settle_s=0.5)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    total_ms = sum(step_ms)
    kern_ms = run.kernel_ms(min(args.steps, 200), flush_l2, stream)
    clk = clocks.stop()

    # end to end through the public API, as a decode step receives its inputs:
    # the step's queries, head weights and lengths and the new tokens' indexer
    # keys and latent rows come from pinned host memory, the rows are appended
    # into the resident caches (dsa_cache_append), the forward runs, and the
    # indices, outputs and LSE are read back.  The appended rows are the rows
    # already at the query positions, so every step computes the same result.
    # Inputs are staged as a server stages them, in one pinned buffer per
    # stream: the indexer's inputs and keys on the main stream, the layers'
    # queries and latent rows on a second stream that the sparse MLA waits for
    # (they upload while the indexer and top-k run); the index set comes back
    # on the second stream while the sparse MLA runs, and the sparse MLA writes
    # the outputs and LSE straight into a pinned host buffer (the device
    # addresses pinned host memory), so they need no copy back.
    from long_context_lightning_gb300 import _lib as lib
    from long_context_lightning_gb300.api import SparseAttention
    seq, pos = wl.query_positions()
    at = torch.cat([W.pool_rows(wl, b, torch.tensor([p_])) for b, p_ in zip(seq, pos)]).to(dev)
    L = spec.n_layers
    part_a = [wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx[at]]
    part_b = [*wl.q, *[kv[at] for kv in wl.kv]]
    part_o = [torch.empty_like(sa.outs[0]) for _ in range(L)] + [torch.empty_like(sa.lses[0]) for _ in range(L)]
    host_a, dev_a, hv_a, dv_a = _staging(part_a, dev)
    host_b, dev_b, _, dv_b = _staging(part_b, dev)
    host_o, dev_o, hv_o, dv_o = _staging(part_o, dev)
    dev_a.copy_(host_a)
    dev_b.copy_(host_b)
    sa_io = SparseAttention(dv_a[0], dv_a[1], dv_a[2], dv_a[3], wl.k_idx, dv_b[:L], wl.kv, spec.d_v, spec.scale,
                            spec.topk, seq_start=wl.seq_start, page_table=wl.page_table, page_size=spec.page_size,
                            outs=hv_o[:L], lses=hv_o[L:])
    new_k, new_c = dv_a[4], dv_b[L:]
    host_idx = torch.empty(sa_io.idx.shape, dtype=torch.int32).pin_memory()
    side = torch.cuda.Stream(dev)
    ev_fork, ev_ready, ev_topk, ev_back = (torch.cuda.Event() for _ in range(4))
    ev_topk.record(stream)  # recorded by the library later on: create the event now
    h2d = host_a.numel() + host_b.numel()
    d2h = host_idx.numel() * 4 + sum(t.numel() * t.element_size() for t in part_o)
    n_e2e = max(3, min(args.steps, 20))

    def e2e_step():
        main = torch.cuda.current_stream(dev)
        ev_fork.record(main)
        side.wait_event(ev_fork)
        with torch.cuda.stream(side):
            dev_b.copy_(host_b, non_blocking=True)
            for layer, c in zip(sa_io.layers, new_c):
                lib.cache_append(sa_io.batch, c, layer.kv, stream=side)
            ev_ready.record(side)
        dev_a.copy_(host_a, non_blocking=True)
        lib.cache_append(sa_io.batch, new_k, sa_io.indexer.k)
        sa_io.forward_overlapped(mla_ready=ev_ready, topk_done=ev_topk)
        side.wait_event(ev_topk)
        with torch.cuda.stream(side):
            host_idx.copy_(sa_io.idx, non_blocking=True)
            ev_back.record(side)
        main.wait_event(ev_back)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    # the step captured once in a CUDA graph (copies from and to pinned host
    # memory included), replayed every step the way a serving loop does
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, capture_error_mode="thread_local"):
        e2e_step()
    for _ in range(2):
        e2e_graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    # what came back equals the device-resident step's results bit for bit
    if not (torch.equal(host_idx, sa.idx.cpu()) and all(torch.equal(h, d.cpu()) for h, d in
                                                        zip(hv_o, list(sa.outs) + list(sa.lses)))):
        raise RuntimeError("decode benchmark: the end-to-end step's results differ from the device step's")
    run.check("decode benchmark")

    # aggregate over ranks: max time
    T = wl.total_q
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dev)
    roof, mla_roof, all_bytes, _ = _roofline(wl, kern_ms, peaks, WORKLOAD)
    wl_cpu = wl.to("cpu")
    del run, sa, sa_io, e2e_graph, host_a, host_b, host_o, dev_a, dev_b, dev_o, hv_a, dv_a, dv_b, hv_o, dv_o
    del new_k, new_c, host_idx, part_a, part_b, part_o
    if rank != 0:
        return
    value = job_throughput(T, world, args.steps, total_ms)
    cpu = _cpu_baseline(spec, wl_cpu, budget_s=8.0) if world == 1 or rank == 0 else None
    del wl_cpu

    # the other workloads: parity cases, timed the same way (rank 0 only, one GPU)
    per_config = {}
    if not args.no_per_config:
        per_config = _per_config(args, dev, stream, flush_l2, peaks)
        per_config["hisparse"] = _hisparse(args, dev, stream, flush_l2)
        per_config["mha"] = _mha_config(args, dev, stream, flush_l2, peaks)

    line = {
        "metric": METRIC, "value": value, "unit": "query tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**_config(spec), "parallelism": f"dp{world} (independent batches per GPU)",
                   "l2": "flushed between timed steps (512 MB write + 256 MB read, outside the timed events)",
                   "cuda_graph": True},
        "roofline": roof,
        "kernels_ms": kern_ms,
        "kernels_ms_source": "separate run of dsa_forward_marked: CUDA events between the four launches on the "
                             "launching stream, L2 flushed before each call; the events stop programmatic "
                             "overlap, so the four means add up to more than ms_per_step",
        "sparse_mla_roofline": mla_roof,
        "step_roofline": _with_nominal({"bound": "hbm", "achieved": all_bytes / (total_ms / args.steps * 1e-3) / 1e9,
                                        "peak": hbm, "unit": "GB/s",
                                        "frac": all_bytes / (total_ms / args.steps * 1e-3) / 1e9 / hbm,
                                        "algorithmic_bytes_per_step": all_bytes}),
        "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "query tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "step": "h2d of the step's indexer inputs, lengths and new indexer keys (one pinned buffer) -> "
                        "dsa_cache_append -> dsa_forward_overlapped, whose sparse MLA waits for the layers' queries "
                        "and new latent rows (a second pinned buffer, uploaded and appended on a second stream "
                        "beside the indexer and top-k) -> d2h of the indices (second stream, beside the sparse "
                        "MLA); outputs and LSE written by the sparse MLA straight into pinned host memory; "
                        "captured once in a CUDA graph and replayed per step; results "
                        "checked bit for bit against the device step's; no L2 flush (the step streams > 349 MB, "
                        "more than the 129 MB L2)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def _scaled(spec, scale):
    """The workload at other sizes (`--scale key=value,...`, for small profiling cases)."""
    if not scale:
        return spec
    kw = {}
    for item in scale.split(","):
        key, val = item.split("=")
        kw[key] = type(getattr(spec, key))(val) if getattr(spec, key) is not None else int(val)
    return spec.scaled(**kw)


def _per_config(args, dev, stream, flush_l2, peaks, names=("tiny", "prefill", "ragged", "indexshare", "csa_flash",
                                                           "csa_pro")):
    out = {}
    steps = max(3, min(args.steps, 20))
    for name in names:
        spec = _scaled(W.SPECS[name], args.scale)
        run = _Run(spec, dev)
        step_ms = run.time_steps(steps, args.warmup, flush_l2, stream)
        kern_ms = run.kernel_ms(steps, flush_l2, stream)
        run.check(name)
        wl = run.wl
        ms = statistics.mean(step_ms)
        T = wl.total_q
        roof, mla_roof, all_bytes, all_flops = _roofline(wl, kern_ms, peaks, name)
        pick, what = CPU_SAMPLE[name]
        queries = pick(T)
        del run
        torch.cuda.empty_cache()
        dt, nq = _oracle_sample(wl, queries, kv_on_device=(name == "indexshare"))
        out[name] = {
            "workload": _config(spec)["workload"] + (f", {spec.n_layers} layers" if spec.n_layers > 1 else "")
                        + (", paged 64-token pages, lengths U{256..16384}" if spec.paged else "")
                        + (f", one cache entry per {spec.compress_ratio} tokens" if spec.compress_ratio > 1 else ""),
            "value": T / (ms * 1e-3), "unit": "query tokens/s" + (" (one query through the 4-layer group)"
                                                                   if spec.n_layers > 1 else ""),
            "ms_per_step": ms, "steps": steps, "kernels_ms": kern_ms, "roofline": roof,
            "sparse_mla_roofline": mla_roof,
            "step": {"algorithmic_bytes": all_bytes, "algorithmic_flops": all_flops,
                     "hbm_frac": all_bytes / (ms * 1e-3) / 1e9 / peaks[0]},
            "cpu_baseline": {"value": nq / dt, "unit": "query tokens/s", "kind": "oracle",
                             "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
                             "sample": f"{nq} queries ({what}), float64 numpy, {dt:.1f} s"},
        }
        del wl
        torch.cuda.empty_cache()
    return out


def _hisparse(args, dev, stream, flush_l2):
    """HiSparse on the decode workload: layer 0's latent pool (32 x 32768 rows)
    in pinned host memory, an HBM slot pool of 262144 rows (a quarter of it).
    Timed with CUDA events on the launching stream, L2 flushed before each:
      cold   the indexer's selection into an empty cache (every row a miss)
      warm   the same selection again (every row a hit)
      step   a chain of selections, each replacing 1/8 of the previous one's
             entries by random positions (the next decode step's top-k overlaps
             the previous one), after the cold fill
    and sparse MLA over the slots beside sparse MLA over the device pool."""
    import oracle
    from long_context_lightning_gb300 import HiSparseCache, _lib
    spec = W.SPECS["decode"]
    run = _Run(spec, dev)
    wl, sa = run.wl, run.sa
    T, k = wl.total_q, spec.topk
    capacity = 262144
    host = wl.kv[0].cpu().pin_memory()
    hc = HiSparseCache(host, capacity, seq_start=wl.seq_start)
    slots = torch.empty((T, k), dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(spec.seed * 1000 + 77)
    n = (wl.seq_lens.to(torch.int64)).view(T, 1)          # one query per sequence, at its last position
    chain = [sa.idx.clone()]
    for _ in range(8):
        nxt = chain[-1].clone()
        fresh = (torch.rand((T, k), generator=g, device=dev) * n).to(torch.int32)
        nxt[:, ::8] = fresh[:, ::8]
        chain.append(nxt)
    ev = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731

    def timed(fn):
        a, b = ev(), ev()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3

    cold, warm, step, step_miss = [], [], [], []
    for rep_i in range(3):
        _lib.hisparse_reset(hc.hs)
        flush_l2(rep_i)
        cold.append(timed(lambda: hc.fetch(sa.batch, chain[0], k, slots)))
        cold_stats = hc.stats()
        flush_l2(rep_i)
        warm.append(timed(lambda: hc.fetch(sa.batch, chain[0], k, slots)))
        for sel in chain[1:]:
            flush_l2(rep_i)
            step.append(timed(lambda: hc.fetch(sa.batch, sel, k, slots)))
            step_miss.append(hc.stats()["misses"])
    run.check("hisparse")
    # sparse MLA over the slots (the last selection) and over the device pool
    hc.fetch(sa.batch, chain[-1], k, slots)
    layer_slots = hc.layer(wl.q[0], spec.d_v, spec.scale)
    out = torch.empty_like(sa.outs[0])
    lse = torch.empty_like(sa.lses[0])
    mla_slots, mla_pool = [], []
    for i in range(5):
        flush_l2(i)
        mla_slots.append(timed(lambda: _lib.sparse_mla_fwd(sa.batch, layer_slots, slots, k, out, lse,
                                                           sa.workspace)))
        flush_l2(i)
        mla_pool.append(timed(lambda: _lib.sparse_mla_fwd(sa.batch, sa.layers[0], chain[-1], k, out, lse,
                                                          sa.workspace)))
    run.check("hisparse sparse MLA")
    # the oracle's LRU bookkeeping on the same trace (host cores)
    wl_cpu = wl.to("cpu", kv_too=False)
    reqs = [oracle.requested_rows(wl_cpu, [r.numpy() for r in sel.cpu()]) for sel in chain]
    lru = oracle.HiSparseLRU(capacity)
    t0 = time.perf_counter()
    for r in reqs:
        lru.step(r)
    dt = time.perf_counter() - t0
    row_bytes = spec.d_qk * 2
    cold_us = statistics.median(cold)
    del run, hc, host
    torch.cuda.empty_cache()
    seq_us, ovl_us = _hisparse_two_layers(dev, stream, flush_l2)
    return {
        "workload": f"decode B={spec.batch} x ctx {spec.ctx_len}: layer-0 latent pool ({spec.batch * spec.ctx_len}"
                    f" rows x {row_bytes} B) in pinned host memory, HBM slot pool of {capacity} rows",
        "cold_fetch_us": cold_us, "cold_misses": cold_stats["misses"],
        "cold_host_to_hbm_GBps": cold_stats["misses"] * row_bytes / (cold_us * 1e-6) / 1e9,
        "warm_fetch_us": statistics.median(warm),
        "step_fetch_us": statistics.median(step), "step_misses_mean": statistics.mean(step_miss),
        "sparse_mla_over_slots_us": statistics.median(mla_slots),
        "sparse_mla_over_pool_us": statistics.median(mla_pool),
        "launches_per_fetch": 7,
        "two_layers_sequential_us": seq_us,
        "two_layers_overlapped_us": ovl_us,
        "two_layers": "decode-like step of two layers sharing one selection: fetch L0, sparse MLA L0, fetch L1, "
                      "sparse MLA L1 on one stream, against L1's fetch on a second stream beside L0's sparse MLA",
        "cpu_baseline": {"value": sum(len(r) for r in reqs) / dt, "unit": "requested rows/s", "kind": "oracle",
                         "cores": 1, "sample": f"LRU bookkeeping of the {len(reqs)}-step trace, python, {dt:.2f} s"},
    }


def _mha_config(args, dev, stream, flush_l2, peaks):
    """MHA mode on its workload (one sequence, context 4608, 3072 queries of
    which 512 see at most 2048 tokens): indexer -> top-k -> per-head
    up-projection of the 4608 latent rows -> attention of every head over its
    selection, replayed from a CUDA graph, L2 flushed between steps."""
    import oracle
    from long_context_lightning_gb300 import SparseMHA, _lib
    from long_context_lightning_gb300 import accounting as A
    spec = _scaled(W.SPECS["mha"], args.scale)
    run = _Run(spec, dev)
    wl, sa = run.wl, run.sa
    T, H, k = wl.total_q, spec.heads, spec.topk
    mha = SparseMHA(wl.cu_seqlens_q, wl.seq_lens, wl.kv[0], wl.w_uk[0], wl.w_uv[0], spec.scale,
                    seq_start=wl.seq_start)
    scores = sa.scores_view()
    out = torch.empty((T, H, 256), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    q = wl.q_mha[0]

    calls = [lambda: _lib.indexer_scores(sa.batch, sa.indexer, scores, sa.workspace),
             lambda: _lib.topk(sa.batch, scores, k, sa.idx, sa.workspace),
             lambda: mha.project(),
             lambda: mha.forward(q, sa.idx, k, out, lse)]
    for c in calls:
        c()
    torch.cuda.synchronize(dev)
    run.check("mha")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        for c in calls:
            c()
    steps = max(3, min(args.steps, 20))
    for _ in range(3):
        graph.replay()
    ev = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731
    step_ms = []
    per = [[] for _ in calls]
    for i in range(steps):
        flush_l2(i)
        a, b = ev(), ev()
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        step_ms.append(a.elapsed_time(b))
    for i in range(steps):
        flush_l2(i)
        marks = [ev() for _ in range(len(calls) + 1)]
        marks[0].record(stream)
        for j, c in enumerate(calls):
            c()
            marks[j + 1].record(stream)
        torch.cuda.synchronize(dev)
        for j in range(len(calls)):
            per[j].append(marks[j].elapsed_time(marks[j + 1]))
    run.check("mha timing")
    names = ["indexer", "topk", "mha_project", "mha_attend"]
    kern_ms = {n: statistics.mean(v) for n, v in zip(names, per)}
    ms = statistics.mean(step_ms)
    hbm, tf_burst, tf_sust, kind = peaks
    shp = _shape(wl)
    att_f = A.mha_attend_flops(shp)
    proj_f = A.mha_project_flops(int(wl.kv[0].shape[0]), H)
    # executed FLOPs of the attention: every 64-key tile up to the last query of a 128-query group
    seq, pos = wl.query_positions()
    exec_f = 0
    for g0 in range(0, T, 128):
        n_last = pos[min(T, g0 + 128) - 1] + 1
        exec_f += 128 * ((n_last + 63) // 64) * 64 * H * (256 + 256) * 2
    att_tf = att_f / (kern_ms["mha_attend"] * 1e-3) / 1e12
    proj_tf = proj_f / (kern_ms["mha_project"] * 1e-3) / 1e12
    cpu = wl.to("cpu")
    t0 = time.perf_counter()
    done = 0
    sample = [T - 1, 0, T // 2, 100]
    while time.perf_counter() - t0 < 2.0 or done < 2:
        t = sample[done % len(sample)]
        sel = oracle.dsa_forward(cpu, queries=[t], layers=[]).idx[t]
        oracle.mha_attention_on_set(cpu, t, 0, sel)
        done += 1
    dt = time.perf_counter() - t0
    del run, mha
    torch.cuda.empty_cache()
    return {
        "workload": f"mha: B=1 x ctx {spec.ctx_len}, {spec.q_per_seq} queries (positions {spec.ctx_len - spec.q_per_seq}"
                    f"..{spec.ctx_len - 1}); indexer {spec.idx_heads}x{spec.idx_dim}; top-k {k}; {H} heads, keys "
                    f"192 up-projected + 64 rope dims, values 256 up-projected, from the 576-dim latent",
        "value": T / (ms * 1e-3), "unit": "query tokens/s", "ms_per_step": ms, "steps": steps,
        "kernels_ms": kern_ms,
        "roofline": _with_nominal({"bound": "tensor", "kernel": "mha_attend", "achieved": att_tf, "peak": tf_sust,
                                   "unit": "TFLOP/s", "frac": att_tf / tf_sust, "traffic": None,
                                   "peak_kind": f"{kind} (bf16 sustained)", "algorithmic_flops_per_launch": att_f,
                                   "executed_flops_per_launch": exec_f,
                                   "executed_tflops": exec_f / (kern_ms["mha_attend"] * 1e-3) / 1e12}),
        "mha_project": {"tflops": proj_tf, "frac": proj_tf / tf_sust, "flops_per_launch": proj_f},
        "cpu_baseline": {"value": done / dt, "unit": "query tokens/s", "kind": "oracle",
                         "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
                         "sample": f"{done} queries (indexer + top-k + per-head up-projection of the selected rows + "
                                   f"64-head attention), float64 numpy, {dt:.1f} s"},
    }


def run_only(args):
    """One workload's per-config entry alone (a small, quick command to profile)."""
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks_all()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    scrub = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def flush_l2(i):  # as in the main run: the lines left in L2 are clean
        flush.fill_(i)
        scrub.sum()

    if args.only == "mha":
        entry = _mha_config(args, dev, stream, flush_l2, peaks)
    elif args.only == "hisparse":
        entry = _hisparse(args, dev, stream, flush_l2)
    else:
        entry = _per_config(args, dev, stream, flush_l2, peaks, names=(args.only,))[args.only]
    print(json.dumps({"only": args.only, "scale": args.scale, "entry": entry}), flush=True)


def _hisparse_two_layers(dev, stream, flush_l2):
    """Two layers of the decode workload, each with its latent pool in pinned
    host memory and an HBM row cache, one selection for both (IndexShare): a
    decode-like step (every eighth entry of the selection replaced) timed with
    the layers in sequence on one stream, and with layer 1's fetch on a second
    stream beside layer 0's sparse MLA (the loads for one layer overlap the
    previous layer's attention)."""
    from long_context_lightning_gb300 import HiSparseCache, _lib
    spec = W.SPECS["decode"].scaled(n_layers=2)
    run = _Run(spec, dev)
    wl, sa = run.wl, run.sa
    T, k = wl.total_q, spec.topk
    hcs = [HiSparseCache(wl.kv[layer].cpu().pin_memory(), 262144, seq_start=wl.seq_start) for layer in range(2)]
    slots = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(2)]
    layers = [hc.layer(wl.q[layer], spec.d_v, spec.scale) for layer, hc in enumerate(hcs)]
    outs = [torch.empty_like(o) for o in sa.outs]
    g = torch.Generator(device=dev)
    g.manual_seed(spec.seed * 1000 + 78)
    n = wl.seq_lens.to(torch.int64).view(T, 1)
    sel = sa.idx.clone()
    side = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731

    def next_sel():
        fresh = (torch.rand((T, k), generator=g, device=dev) * n).to(torch.int32)
        sel[:, ::8] = fresh[:, ::8]

    def mla(layer):
        _lib.sparse_mla_fwd(sa.batch, layers[layer], slots[layer], k, outs[layer], None, sa.workspace)

    def sequential():
        for layer in range(2):
            hcs[layer].fetch(sa.batch, sel, k, slots[layer])
            mla(layer)

    def overlapped():
        hcs[0].fetch(sa.batch, sel, k, slots[0])
        ready = torch.cuda.Event()
        ready.record(stream)
        side.wait_event(ready)
        with torch.cuda.stream(side):
            hcs[1].fetch(sa.batch, sel, k, slots[1], stream=side)
        mla(0)
        done = torch.cuda.Event()
        done.record(side)
        stream.wait_event(done)
        mla(1)

    for fn in (sequential, overlapped):   # fill both caches, warm the code
        fn()
    torch.cuda.synchronize(dev)
    res = {}
    for name, fn in (("sequential", sequential), ("overlapped", overlapped)):
        ts = []
        for i in range(8):
            next_sel()
            flush_l2(i)
            a, b = ev(), ev()
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e3)
        res[name] = statistics.median(ts)
    run.check("hisparse two layers")
    del run, hcs
    torch.cuda.empty_cache()
    return res["sequential"], res["overlapped"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-per-config", action="store_true", help="time the decode headline only")
    ap.add_argument("--only", default=None,
                    help="time one other workload alone (tiny, prefill, ragged, indexshare, csa_flash, csa_pro, mha, "
                         "hisparse) and print its entry; for profiling")
    ap.add_argument("--scale", default=None, help="with --only: workload sizes to change, e.g. ctx_len=32768,q_per_seq=1024")
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
        elif args.only:
            run_only(args)
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
