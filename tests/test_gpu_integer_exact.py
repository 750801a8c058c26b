"""Bit-exact top-k at the full sizes of the four large workloads, on
integer-valued indexer inputs.

With indexer queries and keys integers in [-3, 3] and head weights in
{0.5, 1, 2}, every head's dot product is an integer of magnitude at most
128 * 9 = 1152, and a score is a multiple of 0.5 of magnitude at most
64 * 2 * 1152 = 147456 < 2^23: fp32 (tensor-core accumulation and the fused
epilogue) represents every intermediate exactly, so the scores and hence the
selected set must equal the float64 oracle's bit for bit.  Scores this coarse
tie heavily at the k-th value, so the lowest-position rule is exercised on
every row, across the blocks of a top-k cluster.

These runs take the paths the kernels use at full size: 64 indexer heads and
two 64-dim key blocks, one-query and four-query indexer groups, paged key
tiles, and top-k clusters of up to 16 blocks over 1,048,576-long rows.
"""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import SeqKeys, compare_forward, make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


def _exact_rows(wl_gpu, idx, queries, scores=None):
    """Selected set == oracle top-k, bit for bit; optionally the raw scores too."""
    cpu = wl_gpu.to("cpu", kv_too=False)
    seq, pos = cpu.query_positions()
    k = cpu.spec.topk
    idx = idx.cpu().numpy()
    cache = {}
    tied = 0
    for t in queries:
        b, n = seq[t], pos[t] + 1
        sel = idx[t][idx[t] >= 0]
        if n <= k:
            assert np.array_equal(sel, np.arange(n)), f"query {t}: dense row"
            continue
        if b not in cache:
            cache.clear()
            cache[b] = SeqKeys(cpu, b, int(cpu.seq_lens[b]))
        s = cache[b].scores(cpu, t, n)
        assert np.all(s * 2 == np.round(s * 2)), "integer inputs give multiples of 0.5"
        ref = oracle.topk_select(s, k)
        assert np.array_equal(sel, ref), f"query {t}: top-k differs ({np.setdiff1d(ref, sel)[:5]} missing)"
        theta = np.sort(s)[::-1][k - 1]
        tied += int((s == theta).sum() > 1)
        if scores is not None:
            got = scores[t, :n].double().cpu().numpy()
            assert np.array_equal(got, s), f"query {t}: indexer scores differ"
    return tied


def _integer(name, **kw):
    return W.SPECS[name].scaled(integer_indexer=True, **kw)


def test_decode_full_integer_exact(lib):
    wl = W.make_workload(_integer("decode"), device="cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    T, L = wl.total_q, wl.max_seqlen_k
    scores = torch.full((T, (L + 3) // 4 * 4), float("nan"), dtype=torch.float32, device="cuda")
    lib.indexer_scores(sa.batch, sa.indexer, scores, sa.workspace, skip_dense_k=0)
    assert lib.check_device_error() == lib.DSA_OK
    tied = _exact_rows(wl, idx, range(T), scores=scores)
    assert tied > 0, "no row tied at its k-th score: the tie rule went untested"
    # attention on that exact set, every query
    compare_forward(wl.to("cpu"), idx, outs, lses, range(T), exact_idx=True)


def test_prefill_chunk_full_integer_exact(lib):
    wl = W.make_workload(_integer("prefill"), device="cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    scores = sa.scores_view()          # the fused call's own fp32 scores, still in its workspace
    rng = np.random.default_rng(22)
    sample = sorted({0, 1, 2, 3, 4, 5, 6, 7, 4092, 4093, 4094, 4095, *rng.choice(4096, 20, replace=False).tolist()})
    _exact_rows(wl, idx, sample, scores=scores)


def test_ragged_paged_full_integer_exact(lib):
    wl = W.make_workload(_integer("ragged"), device="cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    _exact_rows(wl, idx, range(wl.total_q), scores=sa.scores_view())


def test_indexshare_1m_integer_exact(lib):
    wl = W.make_workload(_integer("indexshare"), device="cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    _exact_rows(wl, idx, range(wl.total_q), scores=sa.scores_view())
