"""Algorithmic byte and FLOP counts of the DSA forward path (host arithmetic only).

These are the units the roofline numbers are quoted in: what the method must
read, write or compute, not what a given kernel happens to move.

Per sparse query t with causal context n_t = p_t + 1 (> k):
  indexer   bytes  n_t*d_I*2 (indexer keys; shared once per sequence when a
                   chunk of queries of one sequence is scored together)
                   + H_I*d_I*2 (indexer query) + H_I*4 (head weights)
            FLOPs  2*H_I*d_I*n_t
  top-k     bytes  k*4 (selected positions written)
Per query and layer (m_t = min(n_t, k) selected rows):
  sparse MLA bytes m_t*D*2 (gathered latent rows) + H*D*2 (query)
                   + H*D_v*2 (output) + H*4 (LSE) + k*4 (index read)
             FLOPs 2*H*m_t*(D + D_v)   (Q.K over D dims, P.V over D_v dims)

The decode arithmetic intensity of sparse MLA against the gathered rows is
H*(D + D_v)/D FLOP/B; at 64 heads, D = 576, D_v = 512 that is 120.9, the
figure "How GLM5.3 Sparse Attention Affects HBM Memory Usage" (How it works /
Model) gives as 120.8 FLOP/B for 64 query heads.
"""
from __future__ import annotations

import dataclasses
from typing import List


@dataclasses.dataclass
class Shape:
    n: List[int]            # causal context of every query
    seq_of: List[int]       # sequence of every query
    idx_heads: int
    idx_dim: int
    topk: int
    heads: int
    d_qk: int
    d_v: int
    n_layers: int = 1


def indexer_bytes(s: Shape) -> int:
    total = 0
    seen_keys = {}
    for n, b in zip(s.n, s.seq_of):
        if n <= s.topk:
            continue
        seen_keys[b] = max(seen_keys.get(b, 0), n)
        total += s.idx_heads * s.idx_dim * 2 + s.idx_heads * 4
    total += sum(n * s.idx_dim * 2 for n in seen_keys.values())
    return total


def indexer_flops(s: Shape) -> int:
    return sum(2 * s.idx_heads * s.idx_dim * n for n in s.n if n > s.topk)


def topk_bytes(s: Shape) -> int:
    return len(s.n) * s.topk * 4


def mla_bytes(s: Shape, unique_rows_per_seq=None) -> int:
    """Gathered rows counted per query, or once per sequence when the caller
    passes the number of distinct selected rows of each sequence (prefill)."""
    per_q = s.heads * s.d_qk * 2 + s.heads * s.d_v * 2 + s.heads * 4 + s.topk * 4
    total = len(s.n) * per_q
    if unique_rows_per_seq is None:
        total += sum(min(n, s.topk) * s.d_qk * 2 for n in s.n)
    else:
        total += sum(unique_rows_per_seq.values()) * s.d_qk * 2
    return total * s.n_layers


def mla_flops(s: Shape) -> int:
    return sum(2 * s.heads * min(n, s.topk) * (s.d_qk + s.d_v) for n in s.n) * s.n_layers


def decode_intensity(heads: int, d_qk: int, d_v: int) -> float:
    """Sparse-MLA FLOP per byte of gathered latent rows at decode."""
    return heads * (d_qk + d_v) / d_qk


def forward_bytes(s: Shape, unique_rows_per_seq=None) -> int:
    return indexer_bytes(s) + topk_bytes(s) + mla_bytes(s, unique_rows_per_seq)


def forward_flops(s: Shape) -> int:
    return indexer_flops(s) + mla_flops(s)


# MHA mode: every latent row of the context up-projected once into per-head
# keys (d_nope dims + the shared rope dims) and values (d_vh dims), then each
# head attends with its own query over the selection.
def mha_project_flops(rows: int, heads: int, d_latent: int = 512, d_nope: int = 192, d_vh: int = 256) -> int:
    return 2 * rows * heads * (d_nope + d_vh) * d_latent


def mha_project_bytes(rows: int, heads: int, d_row: int = 576, d_latent: int = 512, d_nope: int = 192,
                      d_vh: int = 256, d_head: int = 256) -> int:
    """Latent rows read, projection weights read, per-head key and value rows written."""
    return rows * d_row * 2 + heads * (d_nope + d_vh) * d_latent * 2 + rows * heads * 2 * d_head * 2


def mha_attend_flops(s: Shape, d_head: int = 256, d_vh: int = 256) -> int:
    """Q.K and P.V over the selected positions only (m_t = min(n_t, k) per query)."""
    return sum(2 * s.heads * min(n, s.topk) * (d_head + d_vh) for n in s.n)
