"""Host-side checks that need no GPU: the C ABI library builds, loads and
exports every function include/dsa.h declares; the binding's structs match the
header's; the byte/FLOP accounting and the benchmark's argument handling."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


def _declared_functions():
    hdrs = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]
    names = set()
    for h in hdrs:
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        for m in re.finditer(r"\b(?:dsa_status_t|size_t|const char\*)\s+(dsa_\w+)\s*\(", txt):
            names.add(m.group(1))
    return sorted(names)


def test_library_exports_every_declared_symbol(built):
    lib = ctypes.CDLL(built.LIB_PATH)
    declared = _declared_functions()
    assert len(declared) >= 9
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    assert set(declared) == set(built.EXPORTS), "binding export list out of date with the header"


def test_status_strings_without_gpu(built):
    lib = built.load()
    for s in range(8):
        assert lib.dsa_status_string(s).decode().startswith("DSA_")
    assert "CAPACITY" in lib.dsa_status_string(built.DSA_ERR_CAPACITY).decode()


def test_struct_layout_matches_header(built):
    # sizes/offsets of the ctypes mirrors follow the C layout of dsa.h (LP64)
    assert ctypes.sizeof(built.Cache) == 56
    assert built.Cache.base.offset == 8 and built.Cache.page_table_stride.offset == 48
    assert ctypes.sizeof(built.Batch) == 32
    assert built.Indexer.k.offset == 16 and ctypes.sizeof(built.Indexer) == 80
    assert built.MlaLayer.kv.offset == 8 and built.MlaLayer.scale.offset == 76
    assert ctypes.sizeof(built.HiSparse) == 40
    assert built.HiSparse.slot_pool.offset == 8 and built.HiSparse.state.offset == 32
    assert ctypes.sizeof(built.MhaLayer) == 136
    assert built.MhaLayer.v.offset == 64 and built.MhaLayer.n_heads.offset == 120 and built.MhaLayer.scale.offset == 132


def test_host_validation_without_gpu(built):
    # a NULL batch is rejected before any CUDA call
    lib = built.load()
    assert lib.dsa_workspace_size(None, 2048) == 0
    b = built.Batch(0, 0, 0, 0, None, None)       # num_seqs = 0 is invalid
    assert lib.dsa_workspace_size(ctypes.byref(b), 2048) == 0
    b = built.Batch(2, 2, 1000, 1, 16, 32)         # fake aligned pointers; sizing is host arithmetic
    ws = lib.dsa_workspace_size(ctypes.byref(b), 2048)
    assert ws >= 2 * 1000 * 4
    st = lib.dsa_topk(ctypes.byref(b), None, 1000, 2048, None, 2048, None, 0, None)
    assert st == built.DSA_ERR_INVALID_ARG
    st = lib.dsa_topk(ctypes.byref(b), 16, 1000, 4096, 16, 4096, 16, 1 << 20, None)
    assert st == built.DSA_ERR_UNSUPPORTED


def test_accounting_matches_hand_counts():
    from long_context_lightning_gb300 import accounting as A
    s = A.Shape(n=[32768] * 32, seq_of=list(range(32)), idx_heads=64, idx_dim=128, topk=2048, heads=64,
                d_qk=576, d_v=512)
    # indexer: 32 x (32768 keys x 256 B + 64 x 128 x 2 + 64 x 4)
    assert A.indexer_bytes(s) == 32 * (32768 * 256 + 16384 + 256)
    assert A.indexer_flops(s) == 32 * 2 * 64 * 128 * 32768
    # sparse MLA: 32 x (2048 x 1152 + Q 73728 + O 65536 + LSE 256 + idx 8192)
    assert A.mla_bytes(s) == 32 * (2048 * 1152 + 73728 + 65536 + 256 + 8192)
    assert A.mla_flops(s) == 32 * 2 * 64 * 2048 * 1088
    # dense rows (n <= k) never touch the indexer
    d = A.Shape(n=[100, 3000], seq_of=[0, 1], idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512)
    assert A.indexer_flops(d) == 2 * 64 * 128 * 3000
    # a chunk of queries of one sequence reads the keys once
    p = A.Shape(n=[5000, 5001], seq_of=[0, 0], idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512)
    assert A.indexer_bytes(p) == 5001 * 256 + 2 * (16384 + 256)


def test_bench_reference_line_keys():
    # the reference arm's JSON contract, checked on a tiny budget without a GPU
    import json
    import subprocess
    import sys
    env = dict(os.environ, OPENBLAS_NUM_THREADS="2")
    code = ("import bench, dsa_workloads as W; bench.WORKLOAD='tiny'; "
            "import argparse; a=argparse.Namespace(steps=1, warmup=1); bench.run_reference(a, 0, 1)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "cpu_baseline", "e2e", "config", "dtype"):
        assert k in line
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_host_validation_of_the_later_entry_points(built):
    # every rejection below happens in host code, before any CUDA call
    lib = built.load()
    b = built.Batch(2, 2, 1000, 1, 16, 32)          # fake aligned pointers; nothing is dereferenced
    cache = built.Cache(built.CACHE_CONTIGUOUS, 0, 256, 576, 4000, 64, None, 0)
    # compressed entries: the ratio must be 1 .. max_seqlen_k
    ix = built.Indexer(16, 16, built.Cache(built.CACHE_CONTIGUOUS, 0, 256, 128, 4000, 64, None, 0), 64, 128)
    layer = built.MlaLayer(16, cache, 64, 576, 512, 0.0625)
    arr = (built.MlaLayer * 1)(layer)
    outs = (ctypes.c_void_p * 1)(16)
    for ratio in (0, 1001):
        st = lib.dsa_forward_compressed(ctypes.byref(b), ratio, ctypes.byref(ix), 2048, 1, arr, 16, 2048, outs,
                                        None, 16, 1 << 30, None, None)
        assert st == built.DSA_ERR_INVALID_ARG
    # cache append: no cache, odd row width
    assert lib.dsa_cache_append(ctypes.byref(b), 16, 576, 576, None, None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_cache_append(ctypes.byref(b), 16, 576, 570, ctypes.byref(cache), None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_cache_append(ctypes.byref(b), 8, 576, 576, ctypes.byref(cache), None) == built.DSA_ERR_INVALID_ARG
    # overlapped forward: the same checks as dsa_forward, before any event is touched
    assert lib.dsa_forward_overlapped(ctypes.byref(b), ctypes.byref(ix), 0, 1, arr, 16, 2048, outs, None, 16,
                                      1 << 30, None, None, None) == built.DSA_ERR_UNSUPPORTED
    assert lib.dsa_forward_overlapped(ctypes.byref(b), ctypes.byref(ix), 2048, 0, arr, 16, 2048, outs, None, 16,
                                      1 << 30, None, None, None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_forward_overlapped(ctypes.byref(b), ctypes.byref(ix), 2048, 1, arr, 16, 2048, outs, None, 16,
                                      16, None, None, None) == built.DSA_ERR_WORKSPACE
    # HiSparse sizing and argument checks
    assert lib.dsa_hisparse_state_bytes(0, 100) == 0 and lib.dsa_hisparse_state_bytes(16, 0) == 0
    assert lib.dsa_hisparse_state_bytes(16, 100) >= 12 * 100 + 24 * 16
    assert lib.dsa_hisparse_workspace_size(None, 2048, 16) == 0
    assert lib.dsa_hisparse_workspace_size(ctypes.byref(b), 2048, 0) == 0
    small = lib.dsa_hisparse_workspace_size(ctypes.byref(b), 2048, 16)
    assert 0 < small < lib.dsa_hisparse_workspace_size(ctypes.byref(b), 2048, 1 << 20)   # chunk counts grow
    assert lib.dsa_hisparse_reset(None, None) == built.DSA_ERR_INVALID_ARG
    hs = built.HiSparse(16, 570, 256, 576, 4000, 512)              # row width not a multiple of 8
    assert lib.dsa_hisparse_reset(ctypes.byref(hs), None) == built.DSA_ERR_INVALID_ARG
    hs = built.HiSparse(16, 576, 256, 576, 4000, 512)
    slots = 16
    st = lib.dsa_hisparse_fetch(None, ctypes.byref(b), ctypes.byref(cache), 16, 2048, 2048, slots, 2048, 16,
                                1 << 20, None)
    assert st == built.DSA_ERR_INVALID_ARG
    rows_cache = built.Cache(built.CACHE_ROWS, 0, 256, 576, 4000, None, None, 0)   # a slot pool is not a host pool
    st = lib.dsa_hisparse_fetch(ctypes.byref(hs), ctypes.byref(b), ctypes.byref(rows_cache), 16, 2048, 2048, slots,
                                2048, 16, 1 << 20, None)
    assert st == built.DSA_ERR_INVALID_ARG
    st = lib.dsa_hisparse_fetch(ctypes.byref(hs), ctypes.byref(b), ctypes.byref(cache), 16, 2048, 2048, slots,
                                2048, 16, 64, None)                # workspace too small
    assert st == built.DSA_ERR_WORKSPACE
    # MHA mode: projection arguments, fixed head sizes, context limit, key/value addressing
    assert lib.dsa_mha_project(None, 576, 10, 64, 16, 16, 16, 16, None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_mha_project(16, 500, 10, 64, 16, 16, 16, 16, None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_mha_project(16, 576, 10, 0, 16, 16, 16, 16, None) == built.DSA_ERR_INVALID_ARG
    assert lib.dsa_mha_project(16, 576, 0, 64, 16, 16, 16, 16, None) == built.DSA_OK   # nothing to do
    big = built.Batch(2, 2, 200000, 1, 16, 32)
    assert lib.dsa_mha_workspace_size(ctypes.byref(big)) == 0
    assert lib.dsa_mha_workspace_size(ctypes.byref(b)) > 0
    kc = built.Cache(built.CACHE_CONTIGUOUS, 0, 256, 64 * 256, 4000, 64, None, 0)
    vc = built.Cache(built.CACHE_CONTIGUOUS, 0, 512, 64 * 256, 4000, 64, None, 0)
    ws = lib.dsa_mha_workspace_size(ctypes.byref(b))

    def mha(layer_):
        return lib.dsa_sparse_mha_fwd(ctypes.byref(b), ctypes.byref(layer_), 16, 2048, 2048, 16, None, 16, ws, None)

    assert mha(built.MhaLayer(16, kc, vc, 64, 128, 256, 0.0625)) == built.DSA_ERR_UNSUPPORTED   # head dim
    assert mha(built.MhaLayer(16, kc, vc, 200, 256, 256, 0.0625)) == built.DSA_ERR_UNSUPPORTED  # heads
    other = built.Cache(built.CACHE_CONTIGUOUS, 0, 512, 64 * 256, 4000, 128, None, 0)         # other addressing
    assert mha(built.MhaLayer(16, kc, other, 64, 256, 256, 0.0625)) == built.DSA_ERR_INVALID_ARG
    rows = built.Cache(built.CACHE_ROWS, 0, 256, 64 * 256, 4000, None, None, 0)
    assert mha(built.MhaLayer(16, rows, rows, 64, 256, 256, 0.0625)) == built.DSA_ERR_INVALID_ARG
    st = lib.dsa_sparse_mha_fwd(ctypes.byref(b), ctypes.byref(built.MhaLayer(16, kc, vc, 64, 256, 256, 0.0625)),
                                16, 2048, 2048, 16, None, 16, 64, None)
    assert st == built.DSA_ERR_WORKSPACE


def test_sparse_attention_result_buffers_checked_without_gpu(built):
    # caller-supplied result buffers must have the call's shapes; the check is
    # host-side, before any launch (the tensors here are on the CPU)
    import torch
    import dsa_workloads as W
    from long_context_lightning_gb300 import SparseAttention
    spec = W.SPECS["tiny"]
    wl = W.make_workload(spec)

    def make(**kw):
        return SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, spec.d_v,
                               spec.scale, spec.topk, seq_start=wl.seq_start, **kw)
    T = wl.total_q
    ok = make(idx=torch.empty((T, spec.topk), dtype=torch.int32))
    assert ok.idx.shape == (T, spec.topk)
    with pytest.raises(ValueError):
        make(idx=torch.empty((T, spec.topk + 1), dtype=torch.int32))
    with pytest.raises(ValueError):
        make(idx=torch.empty((T, spec.topk), dtype=torch.int64))
    with pytest.raises(ValueError):
        make(outs=[])


def test_header_is_plain_c_and_links(built, tmp_path):
    # a C99 program against include/dsa.h, linked to the built libdsa.so,
    # calls the host-side entry points without a GPU
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    lib_dir = os.path.dirname(built.load()._name)
    exe = str(tmp_path / "c_abi_check")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                        os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", exe, "-L", lib_dir, "-ldsa",
                        "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
