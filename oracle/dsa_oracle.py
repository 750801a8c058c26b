"""Float64 CPU oracle for the DeepSeek Sparse Attention (DSA) forward path.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import or run this module; the product path never does.
It shares no code with the CUDA library: it takes plain tensors/arrays drawn by
dsa_workloads and writes everything it computes itself, in float64, one query at
a time, in the order the method is described.  A library primitive (matrix
product, sort, exp/log) serves as a step; nothing is blocked, fused or
reordered beyond the definitions below.

What is computed, and where it is defined:

  lightning indexer   I[t, s] = sum_h w[t, h] * max(0, q_I[t, h, :] . k_I[s, :]),
                      for the causal positions s <= p_t.
                      "How GLM5.3 Sparse Attention Affects HBM Memory Usage",
                      How it works / Model, first bullet (down-projected ReLU
                      dot product, summed with weights across heads; selection
                      shared by all attention heads); "DeepSeek Sparse
                      Attention", In the code table: the indexer sums ReLU(q.k) with weights).
  top-k selection     the k causal positions with the largest I[t, .]; when the
                      context holds at most k tokens every token is selected
                      ("How GLM5.3 ...", Model, second bullet: top-k 2048,
                      attention below 2K stays dense).  Equal scores are ordered
                      by lower position first; -0.0 equals +0.0.
  sparse MLA (MQA)    for each head h: z_s = scale * Q[t, h, :D] . C[s, :D] over
                      the selected s; p = softmax(z); O[t, h, :] = sum_s p_s
                      C[s, :D_v]; LSE = log sum_s exp(z_s).  All heads share the
                      one latent row per token ("How GLM5.3 ...", Model, second
                      bullet: sparse MLA in MQA mode).
  IndexShare          one indexer + top-k per group of layers; every layer of
                      the group attends over the same index set ("How GLM5.3
                      ...", How it works / IndexShare: every 4 DSA layers share
                      one indexer and the top-k indices are cached for reuse).
  compressed entries  the same three steps over cache entries that each stand
                      for m consecutive tokens, with top-512 or top-1024
                      entries ("DeepSeek Sparse Attention", In the code: the
                      DeepSeek-V4 indexers score compressed KV entries with
                      ReLU(q.k) scores summed with weights and keep index_topk = 512 or
                      1024).  Reading: entry j stands for tokens m j .. m j +
                      m - 1 and is visible to a query at position p once its
                      block is complete, so the query sees floor((p + 1) / m)
                      entries.
  MHA mode            the same selection; each head's key is the head's
                      up-projection of the latent's first D_v dims followed by
                      the shared rope dims, its value the head's value
                      up-projection; softmax attention per head with the head's
                      own query ("How GLM5.3 ...", Model, second bullet: vLLM
                      switches sparse MLA to MHA mode for about 2K-5K tokens).

Readings where the pages are silent:
  * one indexer key per token, shared by all indexer heads;
  * ReLU per head before weighting; weights unnormalised and may be negative;
  * causality includes the query's own position (n_t = p_t + 1);
  * value = the first D_v dims of the latent row; rope dims enter Q.K only;
  * the returned index set is ascending, padded with -1 to k.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np
import torch


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact bf16 -> float64: a bf16 value is the top 16 bits of a float32."""
    u16 = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f32_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# the three steps, for one query
# ---------------------------------------------------------------------------

def indexer_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Lightning-indexer score of every key for one query.

    q_idx [H_I, d_I], w [H_I], keys [n, d_I] (float64) -> I [n].
    Per head: ReLU of the dot product; then the weighted sum over heads.
    ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", Model, lightning
    indexer bullet.)
    """
    per_head = keys @ q_idx.T                 # [n, H_I]: q_I[h] . k_I[s]
    per_head = np.maximum(per_head, 0.0)      # ReLU per head
    return per_head @ w                       # sum_h w[h] * ReLU(.)


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k largest scores, ties to the lower position, ascending.

    A context of at most k tokens is taken whole ("How GLM5.3 ...", Model:
    attention below 2K tokens stays dense).  -0.0 and +0.0 compare equal.
    """
    n = scores.shape[0]
    if n <= k:
        return np.arange(n, dtype=np.int64)
    pos = np.arange(n, dtype=np.int64)
    order = np.lexsort((pos, -scores))       # primary: score descending; then position ascending
    return np.sort(order[:k])


def sparse_mla(q: np.ndarray, rows: np.ndarray, scale: float, d_v: int):
    """Softmax attention of every head over the selected latent rows.

    q [H, D], rows [m, D] (the selected latent rows) -> O [H, d_v], LSE [H].
    MQA mode: all heads read the same rows; values are rows[:, :d_v].
    An empty selection gives O = 0 and LSE = -inf.
    """
    H = q.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    z = scale * (rows @ q.T)                  # [m, H]
    m = z.max(axis=0)                         # [H]
    e = np.exp(z - m)                         # [m, H]
    Z = e.sum(axis=0)                         # [H]
    O = (e.T @ rows[:, :d_v]) / Z[:, None]    # [H, d_v]
    return O, m + np.log(Z)


# ---------------------------------------------------------------------------
# whole forward over a workload
# ---------------------------------------------------------------------------

def mha_upproject(c_rows: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray):
    """Per-head keys and values of MHA mode from latent rows.

    c_rows [m, D]: the first L dims are the compressed latent, the other D - L
    the rope key every head shares; w_uk [H, d_nope, L]; w_uv [H, d_vh, L].
    Returns K [m, H, d_nope + D - L] with K[s, h] = (w_uk[h] @ c[s, :L], c[s, L:])
    and V [m, H, d_vh] with V[s, h] = w_uv[h] @ c[s, :L].
    """
    L = w_uk.shape[2]
    m, H = c_rows.shape[0], w_uk.shape[0]
    lat = c_rows[:, :L]
    k_nope = np.stack([lat @ w_uk[h].T for h in range(H)], axis=1)      # [m, H, d_nope]
    rope = np.broadcast_to(c_rows[:, None, L:], (m, H, c_rows.shape[1] - L))
    v = np.stack([lat @ w_uv[h].T for h in range(H)], axis=1)           # [m, H, d_vh]
    return np.concatenate([k_nope, rope], axis=2), v


def sparse_mha(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Softmax attention of every head over its own keys and values of the
    selected rows: q [H, d_qk], K [m, H, d_qk], V [m, H, d_vh] -> O [H, d_vh],
    LSE [H].  An empty selection gives O = 0 and LSE = -inf."""
    H = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, V.shape[2])), np.full(H, -np.inf)
    O = np.zeros((H, V.shape[2]))
    lse = np.zeros(H)
    for h in range(H):
        z = scale * (K[:, h, :] @ q[h])       # [m]
        mx = z.max()
        e = np.exp(z - mx)
        Z = e.sum()
        O[h] = (e @ V[:, h, :]) / Z
        lse[h] = mx + math.log(Z)
    return O, lse


def mha_attention_on_set(wl, t: int, layer: int, sel: np.ndarray):
    """MHA-mode attention of query t over the index set `sel` (entries < 0
    skipped): the selected latent rows up-projected per head, then sparse_mha."""
    seq, pos = _query_table(wl)
    sel = np.asarray(sel, dtype=np.int64)
    sel = sel[sel >= 0]
    rows = _rows_of(wl, seq[t], sel)
    pool = wl.kv[layer]
    c = bf16_to_f64(pool[torch.from_numpy(rows).to(pool.device)])
    K, V = mha_upproject(c, bf16_to_f64(wl.w_uk[layer]), bf16_to_f64(wl.w_uv[layer]))
    return sparse_mha(bf16_to_f64(wl.q_mha[layer][t]), K, V, wl.spec.scale)


def _rows_of(wl, b: int, positions: np.ndarray) -> np.ndarray:
    """Pool rows holding tokens `positions` of sequence b (layout lookup)."""
    if wl.page_table is not None:
        ps = wl.spec.page_size
        pt = wl.page_table[b].cpu().numpy().astype(np.int64)
        return pt[positions // ps] * ps + positions % ps
    return int(wl.seq_start[b]) + positions


def _query_table(wl):
    lens = wl.seq_lens.cpu().tolist()
    cu = wl.cu_seqlens_q.cpu().tolist()
    seq, pos = [], []
    for b in range(len(lens)):
        nq = cu[b + 1] - cu[b]
        for i in range(nq):
            seq.append(b)
            pos.append(lens[b] - nq + i)
    return seq, pos


class Forward:
    """Oracle results for selected queries of a workload.

    idx[t]   ascending selected positions (int64, length min(n_t, k))
    out[l][t], lse[l][t]  per layer attention output [H, D_v] and LSE [H]
    scores[t]  float64 indexer scores over the causal context (None when dense)
    indexer_calls  number of indexer evaluations (one per sparse query)
    """

    def __init__(self):
        self.idx = {}
        self.scores = {}
        self.out = []
        self.lse = []
        self.indexer_calls = 0


def dsa_forward(wl, queries: Optional[Sequence[int]] = None, layers: Optional[Sequence[int]] = None,
                keep_scores: bool = False, kv_rows_fetch=None) -> Forward:
    """Run indexer -> top-k -> sparse MLA for the chosen query tokens.

    One indexer evaluation and one top-k per query serve every layer of the
    IndexShare group ("How GLM5.3 ...", IndexShare).  `kv_rows_fetch(layer,
    rows)` may supply latent rows (as a bf16 tensor) when a pool is too large
    to copy whole to the host; by default rows are read from wl.kv[layer].
    """
    spec = wl.spec
    seq, pos = _query_table(wl)
    T = len(seq)
    queries = range(T) if queries is None else list(queries)
    layers = range(spec.n_layers) if layers is None else list(layers)
    res = Forward()
    res.out = [dict() for _ in range(spec.n_layers)]
    res.lse = [dict() for _ in range(spec.n_layers)]
    k_pool = wl.k_idx
    for t in queries:
        b, p = seq[t], pos[t]
        n = visible_entries(p, spec.compress_ratio)       # causal: s <= p (entries of complete blocks)
        if n <= spec.topk:
            sel = np.arange(n, dtype=np.int64)
        else:
            rows = _rows_of(wl, b, np.arange(n, dtype=np.int64))
            keys = bf16_to_f64(k_pool[torch.from_numpy(rows).to(k_pool.device)])
            s = indexer_scores(bf16_to_f64(wl.q_idx[t]), f32_to_f64(wl.w[t]), keys)
            res.indexer_calls += 1
            if keep_scores:
                res.scores[t] = s
            sel = topk_select(s, spec.topk)
        res.idx[t] = sel
        rows = _rows_of(wl, b, sel)
        for layer in layers:
            if kv_rows_fetch is not None:
                c = bf16_to_f64(kv_rows_fetch(layer, rows))
            else:
                pool = wl.kv[layer]
                c = bf16_to_f64(pool[torch.from_numpy(rows).to(pool.device)])
            o, l = sparse_mla(bf16_to_f64(wl.q[layer][t]), c, spec.scale, spec.d_v)
            res.out[layer][t] = o
            res.lse[layer][t] = l
    return res


def cache_append(wl, pool: torch.Tensor, new_rows: torch.Tensor) -> torch.Tensor:
    """A copy of `pool` with the row of every query token written in place.

    Query token t of sequence b sits at position p_t; its row new_rows[t] goes
    to the pool row that holds token p_t of b (page-table or contiguous
    lookup), so that the token is part of its own causal context before the
    indexer scores it (the top-k selector needs the full context in HBM: "How
    GLM5.3 Sparse Attention Affects HBM Memory Usage", What it claims / Model).
    Rows of other tokens are unchanged.
    """
    seq, pos = _query_table(wl)
    out = pool.detach().clone()
    for t, (b, p) in enumerate(zip(seq, pos)):
        r = int(_rows_of(wl, b, np.array([p], dtype=np.int64))[0])
        out[r] = new_rows[t]
    return out


class HiSparseLRU:
    """HBM as a least-recently-used cache of latent rows over host memory
    ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
    HiSparse (SGLang): rows chosen by top-k that are missing from HBM are
    loaded from host DRAM; cold rows are evicted back to DRAM).

    `order` lists the resident rows, least recently used first.  One step takes
    the rows a batch selected (first-request order, repeats ignored):
      * hits are the requested rows already resident, misses the others;
      * the least recently used rows that this step does not request are
        evicted, as many as the misses need (the cache is read-only, so an
        evicted row needs no write-back: host memory holds every row);
      * every requested row becomes most recent: the hits in their previous
        order, then the misses in request order.
    Readings where the pages are silent: the requested rows of one step must
    all fit (capacity >= distinct rows of the step), and rows used in the same
    step keep their relative order as stated above.
    """

    def __init__(self, capacity: int):
        from collections import OrderedDict
        self.capacity = capacity
        self.order = OrderedDict()

    def step(self, requested):
        want = list(dict.fromkeys(int(r) for r in requested))
        want_set = set(want)
        if len(want) > self.capacity:
            raise ValueError("a step requests more distinct rows than the cache holds")
        hits = [r for r in want if r in self.order]
        misses = [r for r in want if r not in self.order]
        n_evict = max(0, len(self.order) + len(misses) - self.capacity)
        evicted = []
        for r in self.order:                       # least recently used first
            if len(evicted) == n_evict:
                break
            if r not in want_set:
                evicted.append(r)
        for r in evicted:
            del self.order[r]
        for r in [r for r in self.order if r in want_set]:
            self.order.move_to_end(r)               # hits, previous relative order
        for r in misses:
            self.order[r] = None                    # then the misses, in request order
        return hits, misses, evicted


def requested_rows(wl, idx_rows) -> list:
    """Pool rows a batch's selection requests, in (query, slot) order: query t's
    row of positions idx_rows[t] (entries < 0 skipped), first occurrences kept."""
    seq, pos = _query_table(wl)
    out = []
    for t in range(len(seq)):
        sel = np.asarray(idx_rows[t], dtype=np.int64)
        sel = sel[sel >= 0]
        out.extend(int(r) for r in _rows_of(wl, seq[t], sel))
    return list(dict.fromkeys(out))


def attention_on_set(wl, t: int, layer: int, sel: np.ndarray, kv_rows_fetch=None):
    """Sparse MLA of query t over an externally supplied index set `sel`
    (used to check the GPU outputs on the GPU's own selection)."""
    seq, pos = _query_table(wl)
    b = seq[t]
    sel = np.asarray(sel, dtype=np.int64)
    sel = sel[sel >= 0]
    rows = _rows_of(wl, b, sel)
    if kv_rows_fetch is not None:
        c = bf16_to_f64(kv_rows_fetch(layer, rows))
    else:
        pool = wl.kv[layer]
        c = bf16_to_f64(pool[torch.from_numpy(rows).to(pool.device)])
    return sparse_mla(bf16_to_f64(wl.q[layer][t]), c, wl.spec.scale, wl.spec.d_v)


def visible_entries(p: int, ratio: int) -> int:
    """Cache entries a query at token position p sees: one per token (ratio 1),
    or the complete blocks of `ratio` tokens."""
    return (p + 1) // ratio


def scores_for_query(wl, t: int) -> np.ndarray:
    """float64 indexer scores of query t over its whole causal context."""
    seq, pos = _query_table(wl)
    b, p = seq[t], pos[t]
    rows = _rows_of(wl, b, np.arange(visible_entries(p, wl.spec.compress_ratio), dtype=np.int64))
    keys = bf16_to_f64(wl.k_idx[torch.from_numpy(rows).to(wl.k_idx.device)])
    return indexer_scores(bf16_to_f64(wl.q_idx[t]), f32_to_f64(wl.w[t]), keys)


def band_check(oracle_scores: np.ndarray, k: int, gpu_sel: np.ndarray, rel_band: float = 1e-3):
    """Compare a selection against the oracle scores with a tie band.

    Every position whose oracle score lies above theta + band must be selected
    and every one below theta - band must not be, where theta is the k-th
    largest oracle score and band = rel_band * |theta|.  Returns a list of
    violations (empty when the selection passes) and theta.
    """
    n = oracle_scores.shape[0]
    sel = np.asarray(gpu_sel, dtype=np.int64)
    sel = sel[sel >= 0]
    problems = []
    if n <= k:
        if not np.array_equal(np.sort(sel), np.arange(n)):
            problems.append("dense row is not 0..n-1")
        return problems, math.nan
    if sel.shape[0] != k:
        problems.append(f"selected {sel.shape[0]} positions, expected {k}")
    if np.unique(sel).shape[0] != sel.shape[0]:
        problems.append("duplicate positions")
    if sel.size and (sel.min() < 0 or sel.max() >= n):
        problems.append("position outside the causal context")
        return problems, math.nan
    theta = np.sort(oracle_scores)[::-1][k - 1]
    band = rel_band * abs(theta)
    chosen = np.zeros(n, dtype=bool)
    chosen[sel] = True
    must = oracle_scores > theta + band
    must_not = oracle_scores < theta - band
    miss = np.nonzero(must & ~chosen)[0]
    extra = np.nonzero(must_not & chosen)[0]
    if miss.size:
        problems.append(f"{miss.size} positions above the band not selected (e.g. {miss[:5].tolist()})")
    if extra.size:
        problems.append(f"{extra.size} positions below the band selected (e.g. {extra[:5].tolist()})")
    return problems, theta
