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
    """

    def __init__(self, cu_seqlens_q: torch.Tensor, seq_lens_k: torch.Tensor, q_idx: torch.Tensor,
                 w: torch.Tensor, k_pool: torch.Tensor, q_layers: Sequence[torch.Tensor],
                 kv_pools: Sequence[torch.Tensor], d_v: int, scale: float, topk: int,
                 seq_start: Optional[torch.Tensor] = None, page_table: Optional[torch.Tensor] = None,
                 page_size: int = 64, total_q: Optional[int] = None, max_seqlen_k: Optional[int] = None,
                 max_q_per_seq: Optional[int] = None, with_lse: bool = True, compress_ratio: int = 1):
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
        self.idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
        self.outs: List[torch.Tensor] = [torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev)
                                         for _ in q_layers]
        self.lses: Optional[List[torch.Tensor]] = (
            [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in q_layers] if with_lse else None)
        ws = _lib.workspace_size(self.batch, topk)
        if ws == 0:
            raise ValueError("invalid batch description")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def forward(self, stream=None):
        """indexer -> top-k -> sparse MLA for every layer; asynchronous on `stream`."""
        _lib.forward(self.batch, self.indexer, self.topk, self.layers, self.idx, self.outs, self.lses,
                     self.workspace, stream, compress_ratio=self.compress_ratio)
        return self.idx, self.outs, self.lses

    def scores_view(self) -> torch.Tensor:
        """The fp32 score matrix the fused call leaves in its workspace ([T, ld]).

        The workspace holds the plan, then room for [T, round_up(max_seqlen_k, 4)]
        fp32 scores; the fused call writes [T, round_up(max entries, 4)] there."""
        ld_tokens = (self.max_seqlen_k + 3) // 4 * 4
        ld = (self.max_seqlen_k // self.compress_ratio + 3) // 4 * 4
        off = self.workspace.numel() - self.total_q * ld_tokens * 4
        return self.workspace[off:off + self.total_q * ld * 4].view(torch.float32).view(self.total_q, ld)
