"""Seeded synthetic workloads for the DeepSeek Sparse Attention (DSA) forward path.

This module only draws inputs: it holds none of the method's arithmetic (no
scores, no selection, no attention).  Both the CUDA path's tests/bench and the
float64 oracle take their inputs from here, and from nowhere else.

Shapes and distributions follow the five workloads the library is measured on:

  tiny        1 sequence, context 512, the last 16 positions are queries;
              indexer 4 heads x 32 dims with integer values in [-3, 3] and
              head weights in {0.5, 1, 2}; top-k 64; attention 8 heads over an
              80-dim latent (64 + 16 rope), values = first 64 dims.
  decode      32 sequences x context 32768, one query each; indexer 64 x 128;
              top-k 2048; 64-head MQA over a 576-dim latent, values 512.
  prefill     1 sequence, context 131072, a chunk of 4096 queries at the end.
  ragged      64 decode queries, contexts uniform in [256, 16384], caches in
              64-token pages with a random page table.
  indexshare  2 decode queries at context 1048576, one indexer shared by 4
              layers, each layer with its own query and latent cache.
  csa_flash   compressed entries (the compressed-sparse-attention layers of
              the DeepSeek-V4 rows in "DeepSeek Sparse Attention", In the code):
              32 decode queries at context 131072 tokens, one entry per 4
              tokens (32768 entries), top-512 entries; indexer 64 x 128,
              64-head MQA over 576-dim entries.
  csa_pro     as csa_flash with top-1024 entries.
  mha         MHA mode ("How GLM5.3 ...", Model: vLLM switches to MHA mode for
              about 2K-5K tokens): 1 sequence, context 4608, the last 3072
              positions are queries (the first 512 of them see at most 2048
              tokens: dense); indexer 64 x 128, top-k 2048; 64 heads whose
              keys (192 no-rope dims up-projected from the 512-dim latent, plus
              the 64 shared rope dims) and values (256 dims up-projected) come
              from the 576-dim latent rows; per-head queries of 256 dims.

The model shapes come from "How GLM5.3 Sparse Attention Affects HBM Memory
Usage" (How it works / Model: 64 query heads, top-k 2048, dense below 2K;
IndexShare: one indexer per 4 layers) and "DeepSeek Sparse Attention" (In the
code: index_topk=2048, index_n_heads=64, index_head_dim=128).  The pages
measure on no dataset; every input is drawn here.

Recipe (device independent up to the device's own generator):
  * every tensor has its own generator, torch.Generator(device).manual_seed(
    seed * 1000 + tensor_id); tensor ids: 0 lengths, 1 page permutation,
    2 indexer queries, 3 head weights, 4 indexer keys, 10+l layer-l queries,
    20+l layer-l latent cache, 30+l layer-l MHA queries, 40+l layer-l key
    up-projection, 50+l layer-l value up-projection.  Any tensor can thus be
    redrawn alone.
  * normal draws are float32 torch.randn scaled by the stated std, then rounded
    to bfloat16 (round to nearest even); integer draws are torch.randint.
  * queries of sequence b are its LAST q_per_seq positions.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

# tensor ids for per-tensor generators
_T_LENS, _T_PAGES, _T_QIDX, _T_W, _T_KIDX, _T_Q, _T_KV = 0, 1, 2, 3, 4, 10, 20
_T_QMHA, _T_WUK, _T_WUV = 30, 40, 50


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    seed: int
    batch: int
    ctx_len: Optional[int]          # fixed context per sequence (None: drawn)
    ctx_range: Optional[tuple]      # inclusive (lo, hi) when drawn
    q_per_seq: int
    idx_heads: int
    idx_dim: int
    topk: int
    heads: int
    d_qk: int
    d_v: int
    scale: float
    n_layers: int = 1
    paged: bool = False
    page_size: int = 64
    integer_indexer: bool = False
    compress_ratio: int = 1         # tokens per cache entry (1: one entry per token)
    mha: bool = False               # MHA mode: per-head keys/values up-projected from the latent
    d_nope: int = 192               # MHA: up-projected no-rope key dims per head (rope = d_qk - d_v)
    d_vh: int = 256                 # MHA: up-projected value dims per head
    q_mha_std: float = 1.0
    idx_std: float = 1.0 / math.sqrt(128.0)
    w_std: float = 1.0 / 8.0
    kv_std: float = 0.05

    def scaled(self, **kw) -> "Spec":
        """Same workload family at other sizes (CPU tests, parity at smaller sizes)."""
        return dataclasses.replace(self, **kw)


SPECS = {
    "tiny": Spec(name="tiny", seed=0, batch=1, ctx_len=512, ctx_range=None, q_per_seq=16,
                 idx_heads=4, idx_dim=32, topk=64, heads=8, d_qk=80, d_v=64,
                 scale=1.0 / math.sqrt(80.0), integer_indexer=True, kv_std=0.1),
    "decode": Spec(name="decode", seed=1, batch=32, ctx_len=32768, ctx_range=None, q_per_seq=1,
                   idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512,
                   scale=1.0 / 16.0),
    "prefill": Spec(name="prefill", seed=2, batch=1, ctx_len=131072, ctx_range=None, q_per_seq=4096,
                    idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512,
                    scale=1.0 / 16.0),
    "ragged": Spec(name="ragged", seed=3, batch=64, ctx_len=None, ctx_range=(256, 16384), q_per_seq=1,
                   idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512,
                   scale=1.0 / 16.0, paged=True),
    "indexshare": Spec(name="indexshare", seed=4, batch=2, ctx_len=1048576, ctx_range=None, q_per_seq=1,
                       idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512,
                       scale=1.0 / 16.0, n_layers=4),
    "csa_flash": Spec(name="csa_flash", seed=5, batch=32, ctx_len=131072, ctx_range=None, q_per_seq=1,
                      idx_heads=64, idx_dim=128, topk=512, heads=64, d_qk=576, d_v=512,
                      scale=1.0 / 16.0, compress_ratio=4),
    "csa_pro": Spec(name="csa_pro", seed=6, batch=32, ctx_len=131072, ctx_range=None, q_per_seq=1,
                    idx_heads=64, idx_dim=128, topk=1024, heads=64, d_qk=576, d_v=512,
                    scale=1.0 / 16.0, compress_ratio=4),
    "mha": Spec(name="mha", seed=7, batch=1, ctx_len=4608, ctx_range=None, q_per_seq=3072,
                idx_heads=64, idx_dim=128, topk=2048, heads=64, d_qk=576, d_v=512,
                scale=1.0 / 16.0, mha=True),
}


@dataclasses.dataclass
class Workload:
    """All inputs of one DSA forward call.

    Layout (row pools shared by every sequence):
      seq_lens     int32 [B]            context length of each sequence
      cu_seqlens_q int32 [B+1]          query offsets; sequence b owns queries
                                        cu[b]..cu[b+1]-1 = its last positions
      q_idx        bf16  [T, H_I, d_I]  indexer queries
      w            fp32  [T, H_I]       indexer head weights
      k_idx        bf16  [R, d_I]       indexer key pool
      q            list of bf16 [T, H, D] per layer
      kv           list of bf16 [R, D]  per-layer latent pools (value = first d_v dims)
      seq_start    int64 [B]            contiguous: token s of b is row seq_start[b]+s
      page_table   int32 [B, P]         paged: token s of b is row
                                        page_table[b, s // page] * page + s % page
    With spec.compress_ratio m > 1 the pools hold one entry per m tokens:
    sequence b of L_b tokens has L_b // m entries (complete blocks), and
    entry j takes the place of token s in the addressing above.
    """
    spec: Spec
    seq_lens: torch.Tensor
    cu_seqlens_q: torch.Tensor
    q_idx: torch.Tensor
    w: torch.Tensor
    k_idx: torch.Tensor
    q: List[torch.Tensor]
    kv: List[torch.Tensor]
    seq_start: Optional[torch.Tensor] = None
    page_table: Optional[torch.Tensor] = None
    q_mha: Optional[List[torch.Tensor]] = None   # MHA mode: per layer bf16 [T, H, d_nope + rope]
    w_uk: Optional[List[torch.Tensor]] = None    # per layer bf16 [H, d_nope, d_v]
    w_uv: Optional[List[torch.Tensor]] = None    # per layer bf16 [H, d_vh, d_v]

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens.max())

    def query_positions(self):
        """(sequence, position) of every query token, as python lists."""
        seq, pos = [], []
        lens = self.seq_lens.tolist()
        cu = self.cu_seqlens_q.tolist()
        for b in range(len(lens)):
            nq = cu[b + 1] - cu[b]
            for i in range(nq):
                seq.append(b)
                pos.append(lens[b] - nq + i)
        return seq, pos

    def to(self, device, kv_too: bool = True) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, seq_lens=mv(self.seq_lens), cu_seqlens_q=mv(self.cu_seqlens_q),
            q_idx=mv(self.q_idx), w=mv(self.w), k_idx=mv(self.k_idx),
            q=[mv(t) for t in self.q], kv=[mv(t) for t in self.kv] if kv_too else self.kv,
            seq_start=mv(self.seq_start), page_table=mv(self.page_table),
            q_mha=None if self.q_mha is None else [mv(t) for t in self.q_mha],
            w_uk=None if self.w_uk is None else [mv(t) for t in self.w_uk],
            w_uv=None if self.w_uv is None else [mv(t) for t in self.w_uv])


def _gen(spec: Spec, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(spec.seed * 1000 + tensor_id)
    return g


def _normal_bf16(shape, std, g, device, chunk_rows=1 << 20):
    """N(0, std^2) rounded to bf16, drawn in row chunks to bound peak memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    inner = shape[1:]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(inner), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (x * std).to(torch.bfloat16)
    return out


def make_workload(spec: Spec, device="cpu", kv_device=None) -> Workload:
    """Draw every input of `spec` on `device` (kv pools on `kv_device`, default `device`)."""
    kv_device = device if kv_device is None else kv_device
    B = spec.batch
    if spec.ctx_len is not None:
        lens = torch.full((B,), spec.ctx_len, dtype=torch.int32)
    else:
        lo, hi = spec.ctx_range
        lens = torch.randint(lo, hi + 1, (B,), generator=_gen(spec, _T_LENS, "cpu"), dtype=torch.int64).to(torch.int32)
    assert int(lens.min()) >= spec.q_per_seq, "every sequence must hold its queries"
    nq = torch.full((B,), spec.q_per_seq, dtype=torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(nq, 0)
    T = int(cu[-1])

    seq_start = page_table = None
    # one pool row per cache entry: a token, or a block of compress_ratio tokens
    n_rows = lens // spec.compress_ratio
    if spec.paged:
        ps = spec.page_size
        npages = [(int(L) + ps - 1) // ps for L in n_rows.tolist()]
        total_pages = sum(npages)
        perm = torch.randperm(total_pages, generator=_gen(spec, _T_PAGES, "cpu")).to(torch.int32)
        page_table = torch.full((B, max(npages)), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(npages):
            page_table[b, :n] = perm[off:off + n]
            off += n
        rows = total_pages * ps
    else:
        seq_start = torch.zeros(B, dtype=torch.int64)
        seq_start[1:] = torch.cumsum(n_rows.to(torch.int64), 0)[:-1]
        rows = int(n_rows.to(torch.int64).sum())

    if spec.integer_indexer:
        q_idx = torch.randint(-3, 4, (T, spec.idx_heads, spec.idx_dim), generator=_gen(spec, _T_QIDX, device),
                              device=device).to(torch.bfloat16)
        choice = torch.randint(0, 3, (T, spec.idx_heads), generator=_gen(spec, _T_W, device), device=device)
        w = torch.tensor([0.5, 1.0, 2.0], dtype=torch.float32, device=device)[choice]
        k_idx = torch.randint(-3, 4, (rows, spec.idx_dim), generator=_gen(spec, _T_KIDX, device),
                              device=device).to(torch.bfloat16)
    else:
        q_idx = _normal_bf16((T, spec.idx_heads, spec.idx_dim), spec.idx_std, _gen(spec, _T_QIDX, device), device)
        w = torch.randn((T, spec.idx_heads), generator=_gen(spec, _T_W, device), device=device,
                        dtype=torch.float32) * spec.w_std
        k_idx = _normal_bf16((rows, spec.idx_dim), spec.idx_std, _gen(spec, _T_KIDX, device), device)

    q, kv = [], []
    for layer in range(spec.n_layers):
        q.append(_normal_bf16((T, spec.heads, spec.d_qk), spec.kv_std, _gen(spec, _T_Q + layer, device), device))
        kv.append(_normal_bf16((rows, spec.d_qk), spec.kv_std, _gen(spec, _T_KV + layer, kv_device), kv_device))

    q_mha = w_uk = w_uv = None
    if spec.mha:
        rope = spec.d_qk - spec.d_v
        q_mha, w_uk, w_uv = [], [], []
        for layer in range(spec.n_layers):
            q_mha.append(_normal_bf16((T, spec.heads, spec.d_nope + rope), spec.q_mha_std,
                                      _gen(spec, _T_QMHA + layer, device), device))
            # unit-gain up-projections: a projected row keeps the latent's scale
            w_uk.append(_normal_bf16((spec.heads, spec.d_nope, spec.d_v), 1.0 / math.sqrt(spec.d_v),
                                     _gen(spec, _T_WUK + layer, device), device))
            w_uv.append(_normal_bf16((spec.heads, spec.d_vh, spec.d_v), 1.0 / math.sqrt(spec.d_v),
                                     _gen(spec, _T_WUV + layer, device), device))

    return Workload(spec=spec, seq_lens=lens.to(device), cu_seqlens_q=cu.to(device), q_idx=q_idx, w=w,
                    k_idx=k_idx, q=q, kv=kv,
                    seq_start=None if seq_start is None else seq_start.to(device),
                    page_table=None if page_table is None else page_table.to(device),
                    q_mha=q_mha, w_uk=w_uk, w_uv=w_uv)


def pool_rows(wl: Workload, b: int, positions: torch.Tensor) -> torch.Tensor:
    """Pool row of token `positions` of sequence b (int64; pure layout lookup)."""
    positions = positions.to(torch.int64)
    if wl.page_table is not None:
        ps = wl.spec.page_size
        pt = wl.page_table[b].to(torch.int64).cpu()
        return pt[positions // ps] * ps + positions % ps
    return int(wl.seq_start[b]) + positions
