"""ctypes binding of libdsa.so (argument marshalling only).

Every compute step runs in the library's CUDA kernels; this module only turns
torch tensors into the pointers and sizes of include/dsa.h and checks the
returned status.  If the library is missing the import of the entry points
fails loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA, DSA_ERR_TIMEOUT, \
    DSA_ERR_BAD_INDEX, DSA_ERR_CAPACITY = range(8)
CACHE_CONTIGUOUS, CACHE_PAGED, CACHE_ROWS = 0, 1, 2
MAX_TOPK = 2048
MAX_LAYERS = 4
MAX_QUERIES = 65535

EXPORTS = ["dsa_status_string", "dsa_check_device_error", "dsa_workspace_size", "dsa_indexer_scores",
           "dsa_topk", "dsa_sparse_mla_fwd", "dsa_forward", "dsa_forward_marked", "dsa_selftest_mma",
           "dsa_selftest_timeout", "dsa_sparse_mla_fwd_noalloc", "dsa_selftest_topk_max_cluster", "dsa_cache_append",
           "dsa_forward_compressed", "dsa_hisparse_state_bytes", "dsa_hisparse_workspace_size", "dsa_hisparse_reset", "dsa_hisparse_fetch",
           "dsa_hisparse_resident", "dsa_hisparse_stats", "dsa_mha_project", "dsa_mha_workspace_size",
           "dsa_sparse_mha_fwd", "dsa_selftest_topk_path", "dsa_forward_overlapped"]
MHA_HEAD_DIM = 256
NOALLOC_MAX_QUERIES = 4096


class Cache(ctypes.Structure):
    _fields_ = [("kind", c_int32), ("page_size", c_int32), ("base", c_void_p), ("row_stride", c_int64),
                ("num_rows", c_int64), ("seq_start", c_void_p), ("page_table", c_void_p),
                ("page_table_stride", c_int64)]


class Batch(ctypes.Structure):
    _fields_ = [("num_seqs", c_int32), ("total_q", c_int32), ("max_seqlen_k", c_int32),
                ("max_q_per_seq", c_int32), ("cu_seqlens_q", c_void_p), ("seq_lens_k", c_void_p)]


class Indexer(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("w", c_void_p), ("k", Cache), ("n_heads", c_int32), ("head_dim", c_int32)]


class MlaLayer(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("kv", Cache), ("n_heads", c_int32), ("d_qk", c_int32), ("d_v", c_int32),
                ("scale", c_float)]


class MhaLayer(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", Cache), ("v", Cache), ("n_heads", c_int32), ("head_dim", c_int32),
                ("v_head_dim", c_int32), ("scale", c_float)]


class HiSparse(ctypes.Structure):
    _fields_ = [("capacity", c_int32), ("row_elems", c_int32), ("slot_pool", c_void_p), ("slot_stride", c_int64),
                ("host_rows", c_int64), ("state", c_void_p)]


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lib = None


def load() -> ctypes.CDLL:
    """Load libdsa.so from the package directory (built by build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libdsa.so is not built ({LIB_PATH}); run long_context_lightning_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [c_int32]
    lib.dsa_check_device_error.restype = c_int32
    lib.dsa_check_device_error.argtypes = [c_void_p]
    lib.dsa_workspace_size.restype = c_size_t
    lib.dsa_workspace_size.argtypes = [POINTER(Batch), c_int32]
    lib.dsa_indexer_scores.restype = c_int32
    lib.dsa_indexer_scores.argtypes = [POINTER(Batch), POINTER(Indexer), c_int32, c_void_p, c_int64, c_void_p,
                                       c_size_t, c_void_p]
    lib.dsa_topk.restype = c_int32
    lib.dsa_topk.argtypes = [POINTER(Batch), c_void_p, c_int64, c_int32, c_void_p, c_int64, c_void_p, c_size_t,
                             c_void_p]
    lib.dsa_sparse_mla_fwd.restype = c_int32
    lib.dsa_sparse_mla_fwd.argtypes = [POINTER(Batch), POINTER(MlaLayer), c_void_p, c_int64, c_int32, c_void_p,
                                       c_void_p, c_void_p, c_size_t, c_void_p]
    lib.dsa_forward.restype = c_int32
    lib.dsa_forward.argtypes = [POINTER(Batch), POINTER(Indexer), c_int32, c_int32, POINTER(MlaLayer), c_void_p,
                                c_int64, POINTER(c_void_p), POINTER(c_void_p), c_void_p, c_size_t, c_void_p]
    lib.dsa_forward_marked.restype = c_int32
    lib.dsa_forward_marked.argtypes = [POINTER(Batch), POINTER(Indexer), c_int32, c_int32, POINTER(MlaLayer),
                                       c_void_p, c_int64, POINTER(c_void_p), POINTER(c_void_p), c_void_p, c_size_t,
                                       c_void_p, POINTER(c_void_p)]
    lib.dsa_sparse_mla_fwd_noalloc.restype = c_int32
    lib.dsa_sparse_mla_fwd_noalloc.argtypes = [POINTER(Batch), POINTER(MlaLayer), c_void_p, c_int64, c_int32,
                                               c_void_p, c_void_p, c_void_p]
    lib.dsa_selftest_mma.restype = c_int32
    lib.dsa_selftest_mma.argtypes = [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p]
    lib.dsa_forward_compressed.restype = c_int32
    lib.dsa_forward_compressed.argtypes = [POINTER(Batch), c_int32, POINTER(Indexer), c_int32, c_int32,
                                           POINTER(MlaLayer), c_void_p, c_int64, POINTER(c_void_p), POINTER(c_void_p),
                                           c_void_p, c_size_t, c_void_p, POINTER(c_void_p)]
    lib.dsa_cache_append.restype = c_int32
    lib.dsa_cache_append.argtypes = [POINTER(Batch), c_void_p, c_int64, c_int32, POINTER(Cache), c_void_p]
    lib.dsa_forward_overlapped.restype = c_int32
    lib.dsa_forward_overlapped.argtypes = [POINTER(Batch), POINTER(Indexer), c_int32, c_int32, POINTER(MlaLayer),
                                           c_void_p, c_int64, POINTER(c_void_p), POINTER(c_void_p), c_void_p,
                                           c_size_t, c_void_p, c_void_p, c_void_p]
    lib.dsa_selftest_topk_max_cluster.restype = c_int32
    lib.dsa_selftest_topk_max_cluster.argtypes = [c_int32]
    lib.dsa_hisparse_state_bytes.restype = c_size_t
    lib.dsa_hisparse_state_bytes.argtypes = [c_int32, c_int64]
    lib.dsa_hisparse_workspace_size.restype = c_size_t
    lib.dsa_hisparse_workspace_size.argtypes = [POINTER(Batch), c_int32, c_int32]
    lib.dsa_hisparse_reset.restype = c_int32
    lib.dsa_hisparse_reset.argtypes = [POINTER(HiSparse), c_void_p]
    lib.dsa_hisparse_fetch.restype = c_int32
    lib.dsa_hisparse_fetch.argtypes = [POINTER(HiSparse), POINTER(Batch), POINTER(Cache), c_void_p, c_int64, c_int32,
                                       c_void_p, c_int64, c_void_p, c_size_t, c_void_p]
    lib.dsa_hisparse_resident.restype = c_int32
    lib.dsa_hisparse_resident.argtypes = [POINTER(HiSparse), c_void_p, c_void_p]
    lib.dsa_hisparse_stats.restype = c_int32
    lib.dsa_hisparse_stats.argtypes = [POINTER(HiSparse), POINTER(c_int32), c_void_p]
    lib.dsa_mha_project.restype = c_int32
    lib.dsa_mha_project.argtypes = [c_void_p, c_int64, c_int64, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p]
    lib.dsa_mha_workspace_size.restype = c_size_t
    lib.dsa_mha_workspace_size.argtypes = [POINTER(Batch)]
    lib.dsa_sparse_mha_fwd.restype = c_int32
    lib.dsa_sparse_mha_fwd.argtypes = [POINTER(Batch), POINTER(MhaLayer), c_void_p, c_int64, c_int32, c_void_p,
                                       c_void_p, c_void_p, c_size_t, c_void_p]
    lib.dsa_selftest_topk_path.restype = c_int32
    lib.dsa_selftest_topk_path.argtypes = [c_int32]
    lib.dsa_selftest_timeout.restype = c_int32
    lib.dsa_selftest_timeout.argtypes = [c_int32, c_void_p]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().dsa_status_string(status).decode()


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------ descriptors ---

def make_batch(cu_seqlens_q: torch.Tensor, seq_lens_k: torch.Tensor, total_q: int, max_seqlen_k: int,
               max_q_per_seq: int) -> Batch:
    """Batch descriptor; the two tensors are int32 device tensors, the ints host copies."""
    assert cu_seqlens_q.dtype == torch.int32 and seq_lens_k.dtype == torch.int32
    return Batch(seq_lens_k.numel(), total_q, max_seqlen_k, max_q_per_seq, _ptr(cu_seqlens_q), _ptr(seq_lens_k))


def make_cache(pool: torch.Tensor, seq_start: Optional[torch.Tensor] = None,
               page_table: Optional[torch.Tensor] = None, page_size: int = 64) -> Cache:
    """Row-pool cache: bf16 [rows, dim] pool plus int64 seq_start, or an int32 [B, P] page table."""
    assert pool.dtype == torch.bfloat16 and pool.dim() == 2 and pool.stride(1) == 1
    if page_table is not None:
        assert page_table.dtype == torch.int32 and page_table.is_contiguous()
        return Cache(CACHE_PAGED, page_size, _ptr(pool), pool.stride(0), pool.shape[0], None, _ptr(page_table),
                     page_table.shape[1])
    assert seq_start is not None and seq_start.dtype == torch.int64
    return Cache(CACHE_CONTIGUOUS, 0, _ptr(pool), pool.stride(0), pool.shape[0], _ptr(seq_start), None, 0)


def make_rows_cache(pool: torch.Tensor) -> Cache:
    """Cache whose selection entries are pool rows themselves (a HiSparse slot pool)."""
    assert pool.dtype == torch.bfloat16 and pool.dim() == 2 and pool.stride(1) == 1
    return Cache(CACHE_ROWS, 0, _ptr(pool), pool.stride(0), pool.shape[0], None, None, 0)


def make_indexer(q_idx: torch.Tensor, w: torch.Tensor, k_cache: Cache) -> Indexer:
    assert q_idx.dtype == torch.bfloat16 and q_idx.is_contiguous() and w.dtype == torch.float32
    return Indexer(_ptr(q_idx), _ptr(w), k_cache, q_idx.shape[1], q_idx.shape[2])


def make_layer(q: torch.Tensor, kv_cache: Cache, d_v: int, scale: float) -> MlaLayer:
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    return MlaLayer(_ptr(q), kv_cache, q.shape[1], q.shape[2], d_v, scale)


# ------------------------------------------------------------ entry points ---

def workspace_size(batch: Batch, topk: int) -> int:
    return int(load().dsa_workspace_size(ctypes.byref(batch), topk))


def indexer_scores(batch: Batch, indexer: Indexer, scores: torch.Tensor, workspace: torch.Tensor,
                   skip_dense_k: int = 0, stream=None):
    assert scores.dtype == torch.float32 and scores.stride(1) == 1
    _check(load().dsa_indexer_scores(ctypes.byref(batch), ctypes.byref(indexer), skip_dense_k, _ptr(scores),
                                     scores.stride(0), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "dsa_indexer_scores")


def topk(batch: Batch, scores: torch.Tensor, k: int, idx: torch.Tensor, workspace: torch.Tensor, stream=None):
    assert idx.dtype == torch.int32 and idx.stride(1) == 1
    _check(load().dsa_topk(ctypes.byref(batch), _ptr(scores), scores.stride(0), k, _ptr(idx), idx.stride(0),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "dsa_topk")


def sparse_mla_fwd(batch: Batch, layer: MlaLayer, idx: torch.Tensor, k: int, out: torch.Tensor,
                   lse: Optional[torch.Tensor], workspace: torch.Tensor, stream=None):
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    _check(load().dsa_sparse_mla_fwd(ctypes.byref(batch), ctypes.byref(layer), _ptr(idx), idx.stride(0), k,
                                     _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "dsa_sparse_mla_fwd")


def sparse_mla_fwd_noalloc(batch: Batch, layer: MlaLayer, idx: torch.Tensor, k: int, out: torch.Tensor,
                           lse: Optional[torch.Tensor], stream=None):
    """sparse_mla_fwd for callers that can pass no workspace (the plan lives in
    a static device array of the library; at most NOALLOC_MAX_QUERIES queries)."""
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    _check(load().dsa_sparse_mla_fwd_noalloc(ctypes.byref(batch), ctypes.byref(layer), _ptr(idx), idx.stride(0), k,
                                             _ptr(out), _ptr(lse), _stream(stream)),
           "dsa_sparse_mla_fwd_noalloc")


def forward(batch: Batch, indexer: Indexer, k: int, layers: Sequence[MlaLayer], idx: torch.Tensor,
            outs: Sequence[torch.Tensor], lses: Optional[Sequence[Optional[torch.Tensor]]],
            workspace: torch.Tensor, stream=None, compress_ratio: int = 1):
    n = len(layers)
    if compress_ratio != 1:
        arr = (MlaLayer * n)(*layers)
        out_ptrs = (c_void_p * n)(*[_ptr(o) for o in outs])
        lse_ptrs = None if lses is None else (c_void_p * n)(*[_ptr(x) for x in lses])
        _check(load().dsa_forward_compressed(ctypes.byref(batch), compress_ratio, ctypes.byref(indexer), k, n, arr,
                                             _ptr(idx), idx.stride(0), out_ptrs, lse_ptrs, _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _stream(stream), None),
               "dsa_forward_compressed")
        return
    arr = (MlaLayer * n)(*layers)
    out_ptrs = (c_void_p * n)(*[_ptr(o) for o in outs])
    lse_ptrs = None if lses is None else (c_void_p * n)(*[_ptr(x) for x in lses])
    _check(load().dsa_forward(ctypes.byref(batch), ctypes.byref(indexer), k, n, arr, _ptr(idx), idx.stride(0),
                              out_ptrs, lse_ptrs, _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream)), "dsa_forward")


def forward_marked(batch: Batch, indexer: Indexer, k: int, layers: Sequence[MlaLayer], idx: torch.Tensor,
                   outs: Sequence[torch.Tensor], lses, workspace: torch.Tensor, marks: Sequence, stream=None,
                   compress_ratio: int = 1):
    """forward() that also records the 5 torch.cuda.Event `marks` between its launches."""
    n = len(layers)
    arr = (MlaLayer * n)(*layers)
    out_ptrs = (c_void_p * n)(*[_ptr(o) for o in outs])
    lse_ptrs = None if lses is None else (c_void_p * n)(*[_ptr(x) for x in lses])
    handles = [m.cuda_event for m in marks]
    if not all(handles):
        raise ValueError("record each torch.cuda.Event once before passing it (torch creates it lazily)")
    ev = (c_void_p * 5)(*handles)
    if compress_ratio != 1:
        _check(load().dsa_forward_compressed(ctypes.byref(batch), compress_ratio, ctypes.byref(indexer), k, n, arr,
                                             _ptr(idx), idx.stride(0), out_ptrs, lse_ptrs, _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _stream(stream), ev),
               "dsa_forward_compressed")
        return
    _check(load().dsa_forward_marked(ctypes.byref(batch), ctypes.byref(indexer), k, n, arr, _ptr(idx),
                                     idx.stride(0), out_ptrs, lse_ptrs, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream), ev),
           "dsa_forward_marked")


def cache_append(batch: Batch, rows: torch.Tensor, cache: Cache, stream=None):
    """Write row t of `rows` (bf16 [T, >= row width]) into `cache` at query token t's position."""
    assert rows.dtype == torch.bfloat16 and rows.stride(1) == 1
    _check(load().dsa_cache_append(ctypes.byref(batch), _ptr(rows), rows.stride(0), rows.shape[1],
                                   ctypes.byref(cache), _stream(stream)), "dsa_cache_append")


def _event(e):
    if e is None:
        return None
    if not e.cuda_event:
        raise ValueError("record each torch.cuda.Event once before passing it (torch creates it lazily)")
    return e.cuda_event


def forward_overlapped(batch: Batch, indexer: Indexer, k: int, layers: Sequence[MlaLayer], idx: torch.Tensor,
                       outs: Sequence[torch.Tensor], lses, workspace: torch.Tensor, stream=None, mla_ready=None,
                       topk_done=None):
    """forward() whose sparse MLA waits for torch.cuda.Event `mla_ready` and which records
    `topk_done` once idx is written (either may be None)."""
    n = len(layers)
    arr = (MlaLayer * n)(*layers)
    out_ptrs = (c_void_p * n)(*[_ptr(o) for o in outs])
    lse_ptrs = None if lses is None else (c_void_p * n)(*[_ptr(x) for x in lses])
    _check(load().dsa_forward_overlapped(ctypes.byref(batch), ctypes.byref(indexer), k, n, arr, _ptr(idx),
                                         idx.stride(0), out_ptrs, lse_ptrs, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream),
                                         _event(mla_ready), _event(topk_done)), "dsa_forward_overlapped")


def hisparse_state_bytes(capacity: int, host_rows: int) -> int:
    return int(load().dsa_hisparse_state_bytes(capacity, host_rows))


def hisparse_workspace_size(batch: Batch, k: int, capacity: int) -> int:
    return int(load().dsa_hisparse_workspace_size(ctypes.byref(batch), k, capacity))


def make_hisparse(slot_pool: torch.Tensor, host_rows: int, state: torch.Tensor) -> HiSparse:
    """Descriptor of an HBM row cache: bf16 [capacity, width] slot pool plus a state buffer."""
    assert slot_pool.dtype == torch.bfloat16 and slot_pool.dim() == 2 and slot_pool.stride(1) == 1
    return HiSparse(slot_pool.shape[0], slot_pool.shape[1], _ptr(slot_pool), slot_pool.stride(0), host_rows,
                    _ptr(state))


def hisparse_reset(hs: HiSparse, stream=None):
    _check(load().dsa_hisparse_reset(ctypes.byref(hs), _stream(stream)), "dsa_hisparse_reset")


def hisparse_fetch(hs: HiSparse, batch: Batch, host_cache: Cache, idx: torch.Tensor, k: int, slots: torch.Tensor,
                   workspace: torch.Tensor, stream=None):
    assert idx.dtype == torch.int32 and idx.stride(1) == 1
    assert slots.dtype == torch.int32 and slots.stride(1) == 1
    _check(load().dsa_hisparse_fetch(ctypes.byref(hs), ctypes.byref(batch), ctypes.byref(host_cache), _ptr(idx),
                                     idx.stride(0), k, _ptr(slots), slots.stride(0), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "dsa_hisparse_fetch")


def hisparse_resident(hs: HiSparse, rows: torch.Tensor, stream=None):
    assert rows.dtype == torch.int32 and rows.is_contiguous() and rows.numel() >= hs.capacity
    _check(load().dsa_hisparse_resident(ctypes.byref(hs), _ptr(rows), _stream(stream)), "dsa_hisparse_resident")


def hisparse_stats(hs: HiSparse, stream=None) -> list:
    out = (c_int32 * 8)()
    _check(load().dsa_hisparse_stats(ctypes.byref(hs), out, _stream(stream)), "dsa_hisparse_stats")
    return list(out)


def mha_project(latent: torch.Tensor, w_uk: torch.Tensor, w_uv: torch.Tensor, k_out: torch.Tensor,
                v_out: torch.Tensor, stream=None):
    """Per-head keys/values of every row of a latent pool (bf16 [rows, >= 576])."""
    assert latent.dtype == torch.bfloat16 and latent.stride(1) == 1
    for t in (w_uk, w_uv, k_out, v_out):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
    _check(load().dsa_mha_project(_ptr(latent), latent.stride(0), latent.shape[0], w_uk.shape[0], _ptr(w_uk),
                                  _ptr(w_uv), _ptr(k_out), _ptr(v_out), _stream(stream)), "dsa_mha_project")


def make_mha_layer(q: torch.Tensor, k_cache: Cache, v_cache: Cache, scale: float) -> MhaLayer:
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    return MhaLayer(_ptr(q), k_cache, v_cache, q.shape[1], q.shape[2], MHA_HEAD_DIM, scale)


def mha_workspace_size(batch: Batch) -> int:
    return int(load().dsa_mha_workspace_size(ctypes.byref(batch)))


def sparse_mha_fwd(batch: Batch, layer: MhaLayer, idx: torch.Tensor, k: int, out: torch.Tensor,
                   lse: Optional[torch.Tensor], workspace: torch.Tensor, stream=None):
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    assert idx.dtype == torch.int32 and idx.stride(1) == 1
    _check(load().dsa_sparse_mha_fwd(ctypes.byref(batch), ctypes.byref(layer), _ptr(idx), idx.stride(0), k,
                                     _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "dsa_sparse_mha_fwd")


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device error status."""
    return int(load().dsa_check_device_error(_stream(stream)))


def selftest_mma(a: torch.Tensor, b: torch.Tensor, d: torch.Tensor, a_mn_major: bool, b_mn_major: bool,
                 swizzle_bytes: int = 128, stream=None):
    _check(load().dsa_selftest_mma(_ptr(a), _ptr(b), _ptr(d), int(a_mn_major), int(b_mn_major), swizzle_bytes,
                                   _stream(stream)), "dsa_selftest_mma")


def selftest_topk_max_cluster(max_cluster: int):
    """Cap the top-k cluster size on the current device (0 restores the default)."""
    _check(load().dsa_selftest_topk_max_cluster(max_cluster), "dsa_selftest_topk_max_cluster")


def selftest_topk_path(candidates: bool):
    """Let the top-k finish from the first digit's candidates (True, the default) or force three passes."""
    _check(load().dsa_selftest_topk_path(1 if candidates else 0), "dsa_selftest_topk_path")


def selftest_timeout(limit_ms: int, stream=None):
    _check(load().dsa_selftest_timeout(limit_ms, _stream(stream)), "dsa_selftest_timeout")
