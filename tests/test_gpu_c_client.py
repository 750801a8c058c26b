"""The fused forward called from a plain-C program through the C ABI alone
(no Python binding in the loop): the test writes a seeded decode problem to
a file, tests/c_forward.c runs dsa_forward on device buffers and writes the
indices, outputs and LSE back, and those are checked against the float64
oracle like every other GPU result."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import dsa_workloads as W
from helpers import compare_forward

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


def _raw(t: torch.Tensor) -> bytes:
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().tobytes()


@pytest.mark.parametrize("kw", [dict(batch=3, ctx_len=3000), dict(batch=5, ctx_len=1900)])
def test_c_client_forward_matches_oracle(lib, tmp_path, kw):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    spec = W.SPECS["decode"].scaled(**kw)
    wl = W.make_workload(spec)
    T, R = wl.total_q, wl.k_idx.shape[0]
    hdr = np.array([spec.batch, T, int(wl.seq_lens.max()), 1, spec.idx_heads, spec.idx_dim, spec.heads, spec.d_qk,
                    spec.d_v, spec.topk, R], dtype=np.int64).tobytes() + np.array([spec.scale], np.float64).tobytes()
    src = tmp_path / "problem.bin"
    src.write_bytes(hdr + b"".join(_raw(x) for x in (wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx,
                                                     wl.q[0], wl.kv[0], wl.seq_start)))
    lib_dir = os.path.dirname(lib.load()._name)
    exe = str(tmp_path / "c_forward")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                        CUDA + "/include", os.path.join(ROOT, "tests", "c_forward.c"), "-o", exe, "-L", lib_dir,
                        "-ldsa", "-L", CUDA + "/lib64", "-lcudart", "-Wl,-rpath," + lib_dir,
                        "-Wl,-rpath," + CUDA + "/lib64"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    dst = tmp_path / "result.bin"
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
    raw = dst.read_bytes()
    n_idx, n_out = T * spec.topk * 4, T * spec.heads * spec.d_v * 2
    idx = torch.frombuffer(bytearray(raw[:n_idx]), dtype=torch.int32).view(T, spec.topk)
    out = torch.frombuffer(bytearray(raw[n_idx:n_idx + n_out]), dtype=torch.int16).view(torch.bfloat16)
    lse = torch.frombuffer(bytearray(raw[n_idx + n_out:]), dtype=torch.float32).view(T, spec.heads)
    compare_forward(wl, idx, [out.view(T, spec.heads, spec.d_v)], [lse], range(T))
