"""Python front end of the DSA forward path: holds the descriptors and buffers
of one problem and calls the C ABI.  Buffers are torch tensors (device memory
and streams are PyTorch's); every step of the path runs in libdsa.so.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import _lib


class SparseAttention:
    """One DSA problem: a ragged batch, one indexer and an IndexShare group of
    1..4 sparse-MLA layers that share its top-k positions.

    cu_seqlens_q  int32 [B+1] device; seq_lens_k int32 [B] device
    q_idx         bf16 [T, H_I, d_I]; w fp32 [T, H_I]
    k_pool        bf16 [rows, d_I] indexer-key pool
    q_layers      per layer bf16 [T, H, D]; kv_pools per layer bf16 [rows, D]
    seq_start     int64 [B] (contiguous pools) or page_table int32 [B, P] (paged)
    compress_ratio  tokens per cache entry (pools of compressed entries; 1: one row per token)
    idx, outs, lses  optional result buffers (int32 [T, topk]; per layer bf16 [T, H, d_v] and
                  fp32 [T, H]); new ones are allocated when omitted
    """

    def __init__(self, cu_seqlens_q: torch.Tensor, seq_lens_k: torch.Tensor, q_idx: torch.Tensor,
                 w: torch.Tensor, k_pool: torch.Tensor, q_layers: Sequence[torch.Tensor],
                 kv_pools: Sequence[torch.Tensor], d_v: int, scale: float, topk: int,
                 seq_start: Optional[torch.Tensor] = None, page_table: Optional[torch.Tensor] = None,
                 page_size: int = 64, total_q: Optional[int] = None, max_seqlen_k: Optional[int] = None,
                 max_q_per_seq: Optional[int] = None, with_lse: bool = True, compress_ratio: int = 1,
                 idx: Optional[torch.Tensor] = None, outs: Optional[Sequence[torch.Tensor]] = None,
                 lses: Optional[Sequence[torch.Tensor]] = None):
        dev = q_idx.device
        self.topk = topk
        self.compress_ratio = compress_ratio
        nq = (cu_seqlens_q[1:] - cu_seqlens_q[:-1])
        self.total_q = int(cu_seqlens_q[-1]) if total_q is None else total_q
        self.max_seqlen_k = int(seq_lens_k.max()) if max_seqlen_k is None else max_seqlen_k
        self.max_q_per_seq = int(nq.max()) if max_q_per_seq is None else max_q_per_seq
        self._keep = [cu_seqlens_q, seq_lens_k, q_idx, w, k_pool, *q_layers, *kv_pools, seq_start, page_table]
        self.batch = _lib.make_batch(cu_seqlens_q, seq_lens_k, self.total_q, self.max_seqlen_k, self.max_q_per_seq)
        self.indexer = _lib.make_indexer(q_idx, w, _lib.make_cache(k_pool, seq_start, page_table, page_size))
        self.layers = [_lib.make_layer(q, _lib.make_cache(kv, seq_start, page_table, page_size), d_v, scale)
                       for q, kv in zip(q_layers, kv_pools)]
        T = self.total_q
        H = q_layers[0].shape[1]
        # result buffers: the caller's (e.g. views of one staging buffer) or new ones
        self.idx = torch.empty((T, topk), dtype=torch.int32, device=dev) if idx is None else idx
        self.outs: List[torch.Tensor] = (
            [torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev) for _ in q_layers] if outs is None
            else list(outs))
        if lses is not None:
            self.lses: Optional[List[torch.Tensor]] = list(lses)
        else:
            self.lses = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in q_layers] if with_lse else None
        if tuple(self.idx.shape) != (T, topk) or self.idx.dtype != torch.int32 or len(self.outs) != len(q_layers):
            raise ValueError("idx must be int32 [total_q, topk] and outs one [total_q, heads, d_v] per layer")
        ws = _lib.workspace_size(self.batch, topk)
        if ws == 0:
            raise ValueError("invalid batch description")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def forward(self, stream=None):
        """indexer -> top-k -> sparse MLA for every layer; asynchronous on `stream`."""
        _lib.forward(self.batch, self.indexer, self.topk, self.layers, self.idx, self.outs, self.lses,
                     self.workspace, stream, compress_ratio=self.compress_ratio)
        return self.idx, self.outs, self.lses

    def forward_overlapped(self, stream=None, mla_ready=None, topk_done=None):
        """forward() for a step whose layer inputs arrive while it runs: the sparse MLA waits
        for torch.cuda.Event `mla_ready` (queries uploaded, latent rows appended on another
        stream), and `topk_done` is recorded once the index set is written.  Tokens only."""
        if self.compress_ratio != 1:
            raise ValueError("forward_overlapped serves token caches (compress_ratio 1)")
        _lib.forward_overlapped(self.batch, self.indexer, self.topk, self.layers, self.idx, self.outs, self.lses,
                                self.workspace, stream, mla_ready, topk_done)
        return self.idx, self.outs, self.lses

    def scores_view(self) -> torch.Tensor:
        """The fp32 score matrix the fused call leaves in its workspace ([T, ld]).

        The workspace holds the plan, then room for [T, round_up(max_seqlen_k, 4)]
        fp32 scores; the fused call writes [T, round_up(max entries, 4)] there."""
        ld_tokens = (self.max_seqlen_k + 3) // 4 * 4
        ld = (self.max_seqlen_k // self.compress_ratio + 3) // 4 * 4
        off = self.workspace.numel() - self.total_q * ld_tokens * 4
        return self.workspace[off:off + self.total_q * ld * 4].view(torch.float32).view(self.total_q, ld)


class HiSparseCache:
    """HBM slot pool holding the most recently used rows of one layer's latent
    pool, which lives in pinned host memory.

    fetch() makes every row a selection asks for resident (misses copied from
    host memory, least recently used rows that the step does not ask for
    evicted) and writes the slot of each selected entry; layer() gives the
    sparse-MLA descriptor that reads those slots.  The host pool keeps its
    addressing (seq_start or page_table, as for SparseAttention).
    """

    def __init__(self, host_pool: torch.Tensor, capacity: int, seq_start: Optional[torch.Tensor] = None,
                 page_table: Optional[torch.Tensor] = None, page_size: int = 64, device=None):
        if not host_pool.is_pinned():
            raise ValueError("the host pool must be pinned host memory (tensor.pin_memory())")
        device = torch.device("cuda") if device is None else torch.device(device)
        self.host_pool = host_pool
        self.host_cache = _lib.make_cache(host_pool, seq_start, page_table, page_size)
        self.slot_pool = torch.empty((capacity, host_pool.shape[1]), dtype=torch.bfloat16, device=device)
        self.state = torch.empty(_lib.hisparse_state_bytes(capacity, host_pool.shape[0]), dtype=torch.uint8,
                                 device=device)
        self.hs = _lib.make_hisparse(self.slot_pool, host_pool.shape[0], self.state)
        self.rows_cache = _lib.make_rows_cache(self.slot_pool)
        self._keep = [seq_start, page_table]
        self._ws: Optional[torch.Tensor] = None
        _lib.hisparse_reset(self.hs)

    def fetch(self, batch, idx: torch.Tensor, k: int, slots: torch.Tensor, workspace: Optional[torch.Tensor] = None,
              stream=None):
        """Asynchronous on `stream`: slots[t, j] = slot of idx[t, j]'s row (-1 where idx is -1).
        Without `workspace` the cache keeps one of its own (grown as needed)."""
        if workspace is None:
            need = _lib.hisparse_workspace_size(batch, k, self.hs.capacity)
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(need, dtype=torch.uint8, device=self.slot_pool.device)
            workspace = self._ws
        _lib.hisparse_fetch(self.hs, batch, self.host_cache, idx, k, slots, workspace, stream)
        return slots

    def layer(self, q: torch.Tensor, d_v: int, scale: float):
        """Sparse-MLA layer descriptor over the slot pool (pass the slots as its index set)."""
        return _lib.make_layer(q, self.rows_cache, d_v, scale)

    def resident(self) -> List[int]:
        """Resident host rows, least recently used first."""
        rows = torch.empty(self.hs.capacity, dtype=torch.int32, device=self.slot_pool.device)
        _lib.hisparse_resident(self.hs, rows)
        return [r for r in rows.cpu().tolist() if r >= 0]

    def stats(self) -> dict:
        s = _lib.hisparse_stats(self.hs)
        return dict(steps=s[0], requested=s[1], hits=s[2], misses=s[3], evicted=s[4], overflow=s[5])


class SparseMHA:
    """MHA mode over a short context: the latent pool up-projected once into
    per-head keys and values (`project`), then attention of every head over
    each query's top-k selection (`forward`).  The per-head caches keep the
    latent pool's row numbers and addressing (seq_start or page_table)."""

    def __init__(self, cu_seqlens_q: torch.Tensor, seq_lens_k: torch.Tensor, latent_pool: torch.Tensor,
                 w_uk: torch.Tensor, w_uv: torch.Tensor, scale: float, seq_start: Optional[torch.Tensor] = None,
                 page_table: Optional[torch.Tensor] = None, page_size: int = 64):
        dev = latent_pool.device
        H = w_uk.shape[0]
        rows = latent_pool.shape[0]
        nq = (cu_seqlens_q[1:] - cu_seqlens_q[:-1]).cpu()
        self.total_q = int(cu_seqlens_q[-1])
        self.batch = _lib.make_batch(cu_seqlens_q, seq_lens_k, self.total_q, int(seq_lens_k.max()), int(nq.max()))
        self.latent, self.w_uk, self.w_uv, self.scale = latent_pool, w_uk, w_uv, scale
        self.k_pool = torch.empty((rows, H * _lib.MHA_HEAD_DIM), dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.empty((rows, H * _lib.MHA_HEAD_DIM), dtype=torch.bfloat16, device=dev)
        self.k_cache = _lib.make_cache(self.k_pool, seq_start, page_table, page_size)
        self.v_cache = _lib.make_cache(self.v_pool, seq_start, page_table, page_size)
        self._keep = [cu_seqlens_q, seq_lens_k, seq_start, page_table]
        self.workspace = torch.empty(_lib.mha_workspace_size(self.batch), dtype=torch.uint8, device=dev)

    def project(self, stream=None):
        """Per-head keys and values of every latent row; asynchronous on `stream`."""
        _lib.mha_project(self.latent, self.w_uk, self.w_uv, self.k_pool, self.v_pool, stream)

    def forward(self, q: torch.Tensor, idx: torch.Tensor, k: int, out: torch.Tensor,
                lse: Optional[torch.Tensor] = None, stream=None):
        """out[t, h] = attention of q[t, h] (bf16 [T, H, 256]) over the selection idx[t]."""
        layer = _lib.make_mha_layer(q, self.k_cache, self.v_cache, self.scale)
        _lib.sparse_mha_fwd(self.batch, layer, idx, k, out, lse, self.workspace, stream)
        return out, lse
