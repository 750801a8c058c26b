"""Shared test helpers: run the CUDA path on a workload and compare it with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import dsa_workloads as W
import oracle

OUT_MAX_REL = 1e-2    # max |err| <= 1e-2 * max |ref|
OUT_MEAN_REL = 1e-3   # mean |err| <= 1e-3 * max |ref|
BAND_REL = 1e-3       # selection band around the k-th oracle score


def make_sa(wl, with_lse=True):
    from long_context_lightning_gb300 import SparseAttention
    s = wl.spec
    return SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, s.d_v, s.scale,
                           s.topk, seq_start=wl.seq_start, page_table=wl.page_table, page_size=s.page_size,
                           with_lse=with_lse, compress_ratio=s.compress_ratio)


def sel_of(row: np.ndarray) -> np.ndarray:
    return row[row >= 0]


def check_output(got: np.ndarray, ref: np.ndarray, what: str):
    """got [H, D_v] (from bf16), ref float64 [H, D_v]."""
    err = np.abs(got.astype(np.float64) - ref)
    m = np.abs(ref).max()
    assert err.max() <= OUT_MAX_REL * m, f"{what}: max err {err.max():.3e} > {OUT_MAX_REL} * {m:.3e}"
    assert err.mean() <= OUT_MEAN_REL * m, f"{what}: mean err {err.mean():.3e} > {OUT_MEAN_REL} * {m:.3e}"


def check_lse(got: np.ndarray, ref: np.ndarray, what: str):
    np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-4, err_msg=what)


class SeqKeys:
    """float64 indexer keys of one sequence, decoded once with the oracle's own
    bf16 -> float64 conversion, so that many queries of that sequence are
    scored by oracle.indexer_scores without re-reading the pool each time."""

    def __init__(self, wl, b, n):
        rows = W.pool_rows(wl, b, torch.arange(n))
        self.b = b
        self.keys = oracle.bf16_to_f64(wl.k_idx[rows.to(wl.k_idx.device)])

    def scores(self, wl, t, n):
        return oracle.indexer_scores(oracle.bf16_to_f64(wl.q_idx[t]), oracle.f32_to_f64(wl.w[t]), self.keys[:n])


def compare_forward(wl, idx, outs, lses, queries, exact_idx=False, kv_rows_fetch=None, seq_keys=None):
    """Compare the GPU result of `queries` with the oracle.

    Indices: bit-exact when `exact_idx` (integer indexer inputs), else the band
    rule.  Outputs/LSE: oracle attention over the GPU's own index set, for every
    layer (near-tie swaps inside the band change attention legitimately).
    `seq_keys` (a SeqKeys of the queries' one sequence) speeds up scoring many
    queries of one long sequence.
    """
    spec = wl.spec
    seq, pos = wl.query_positions()
    idx = idx.cpu().numpy()
    for t in queries:
        n = oracle.visible_entries(pos[t], spec.compress_ratio)
        row = idx[t]
        sel = sel_of(row)
        assert np.all(np.diff(sel) > 0), f"query {t}: selection not ascending/distinct"
        assert np.all(row[len(sel):] == -1), f"query {t}: padding"
        if n <= spec.topk:
            assert np.array_equal(sel, np.arange(n)), f"query {t}: dense row"
        else:
            if seq_keys is not None and seq_keys.b == seq[t]:
                s = seq_keys.scores(wl, t, n)
            else:
                s = oracle.scores_for_query(wl, t)
            if exact_idx:
                assert np.array_equal(sel, oracle.topk_select(s, spec.topk)), f"query {t}: top-k differs"
            else:
                problems, _ = oracle.band_check(s, spec.topk, sel, BAND_REL)
                assert not problems, f"query {t}: {problems}"
        for layer in range(spec.n_layers):
            o, l = oracle.attention_on_set(wl, t, layer, sel, kv_rows_fetch=kv_rows_fetch)
            H = spec.heads
            check_output(outs[layer][t].float().cpu().numpy(), o[:H], f"query {t} layer {layer}")
            if lses is not None:
                check_lse(lses[layer][t].cpu().numpy(), l[:H], f"query {t} layer {layer} lse")
