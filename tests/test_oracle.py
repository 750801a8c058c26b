"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test checks a closed form, an invariant, a special case that reduces to a
library routine (torch's scaled_dot_product_attention in float64), a defining
property checked by brute force, or a figure printed on the pages.  Each is
chosen so that a plausible mistake (ReLU after the head sum, a transposed
operand, a dropped scale, values taken from the wrong dims, ties broken the
wrong way, an off-by-one in causality) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from long_context_lightning_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- indexer ---

def test_indexer_unit_query_reads_one_key_column():
    # one head, weight 1, q = e_c  ->  I[s] = max(0, k[s, c])
    keys = rng.standard_normal((50, 16))
    for c in (0, 7, 15):
        q = np.zeros((1, 16)); q[0, c] = 1.0
        got = oracle.indexer_scores(q, np.array([1.0]), keys)
        np.testing.assert_array_equal(got, np.maximum(keys[:, c], 0.0))


def test_indexer_relu_is_per_head_before_weighting():
    # heads q and -q with weights (1, 1): relu(x) + relu(-x) = |x|.
    # A ReLU applied after the head sum would give relu(0) = 0 instead.
    d = 8
    a = rng.integers(-5, 6, size=d).astype(np.float64)
    v = rng.integers(-5, 6, size=d).astype(np.float64)
    keys = np.diag(a)                       # q . k_s = v[s] * a[s] without a matmul
    q = np.stack([v, -v])
    got = oracle.indexer_scores(q, np.array([1.0, 1.0]), keys)
    np.testing.assert_array_equal(got, np.abs(v * a))
    # a negative weight flips the sign of that head's (non-negative) term
    got = oracle.indexer_scores(v[None, :], np.array([-2.0]), keys)
    np.testing.assert_array_equal(got, -2.0 * np.maximum(v * a, 0.0))


def test_indexer_linear_in_weights_homogeneous_in_query_equivariant_in_keys():
    q = rng.standard_normal((6, 12)); keys = rng.standard_normal((40, 12))
    w1 = rng.standard_normal(6); w2 = rng.standard_normal(6)
    i1 = oracle.indexer_scores(q, w1, keys); i2 = oracle.indexer_scores(q, w2, keys)
    np.testing.assert_allclose(oracle.indexer_scores(q, w1 + w2, keys), i1 + i2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.indexer_scores(2.0 * q, w1, keys), 2.0 * i1, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(40)
    np.testing.assert_allclose(oracle.indexer_scores(q, w1, keys[perm]), i1[perm], rtol=1e-12, atol=1e-12)


def test_indexer_exact_on_integer_inputs_brute_force():
    # tiny workload: integer q, k in [-3, 3], weights in {0.5, 1, 2}: exact
    # rational arithmetic with python ints must agree bit for bit.
    wl = W.make_workload(W.SPECS["tiny"])
    t = 3
    s = oracle.scores_for_query(wl, t)
    q = wl.q_idx[t].float().tolist(); w = wl.w[t].tolist()
    seq, pos = wl.query_positions()
    for sp in (0, 1, 100, pos[t]):
        k = wl.k_idx[int(wl.seq_start[0]) + sp].float().tolist()
        exact = 0.0
        for h in range(len(q)):
            dot = sum(int(a) * int(b) for a, b in zip(q[h], k))
            exact += w[h] * max(0, dot)
        assert s[sp] == exact
    assert np.all(s * 2 == np.round(s * 2))            # multiples of 0.5


# ------------------------------------------------------------------ top-k ---

def _check_topk_property(scores, k, sel):
    n = scores.shape[0]
    sel = np.asarray(sel)
    assert np.all(np.diff(sel) > 0), "ascending, distinct"
    if n <= k:
        assert np.array_equal(sel, np.arange(n)); return
    assert sel.shape[0] == k
    chosen = np.zeros(n, bool); chosen[sel] = True
    # brute force over all (selected, unselected) pairs
    for s in np.nonzero(chosen)[0]:
        for u in np.nonzero(~chosen)[0]:
            assert scores[s] > scores[u] or (scores[s] == scores[u] and s < u)


def test_topk_defining_property_with_many_ties():
    for n, k in ((40, 7), (64, 64), (65, 64), (100, 1), (30, 50)):
        scores = rng.integers(-3, 4, size=n).astype(np.float64)
        _check_topk_property(scores, k, oracle.topk_select(scores, k))


def test_topk_permutation_closed_form():
    n, k = 1000, 37
    scores = rng.permutation(n).astype(np.float64)
    sel = oracle.topk_select(scores, k)
    np.testing.assert_array_equal(sel, np.nonzero(scores >= n - k)[0])


def test_topk_all_equal_takes_lowest_positions_and_signed_zero_ties():
    np.testing.assert_array_equal(oracle.topk_select(np.full(100, 2.5), 10), np.arange(10))
    z = np.zeros(20); z[::2] = -0.0                 # -0.0 == +0.0: ties by position
    assert np.signbit(z[0])
    np.testing.assert_array_equal(oracle.topk_select(z, 5), np.arange(5))


def test_topk_dense_when_context_fits():
    # "attention below 2K tokens stays dense": n <= k selects every position
    np.testing.assert_array_equal(oracle.topk_select(rng.standard_normal(2048), 2048), np.arange(2048))
    assert oracle.topk_select(rng.standard_normal(2049), 2048).shape == (2048,)


# ------------------------------------------------------------- sparse MLA ---

def _sdpa_f64(q, rows, scale, d_v, mask=None):
    # torch's attention routine in float64: q [H, D], keys = rows, values = rows[:, :d_v]
    Q = torch.from_numpy(q)[None, :, None, :]                      # [1, H, 1, D]
    K = torch.from_numpy(rows)[None, None].expand(1, q.shape[0], -1, -1)
    V = torch.from_numpy(rows[:, :d_v].copy())[None, None].expand(1, q.shape[0], -1, -1)
    am = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=am, scale=scale)
    return out[0, :, 0, :].numpy()


def test_mla_dense_case_equals_library_attention():
    # k >= n: the selection is the whole causal context, so sparse MLA must be
    # dense MQA softmax attention
    H, D, Dv, n = 8, 80, 64, 37
    q = rng.standard_normal((H, D)); rows = rng.standard_normal((n, D))
    o, lse = oracle.sparse_mla(q, rows, 1 / math.sqrt(D), Dv)
    np.testing.assert_allclose(o, _sdpa_f64(q, rows, 1 / math.sqrt(D), Dv), rtol=1e-12, atol=1e-12)
    z = (rows @ q.T) / math.sqrt(D)
    np.testing.assert_allclose(lse, np.log(np.exp(z).sum(0)), rtol=1e-12)


def test_mla_equals_dense_attention_with_additive_mask():
    # the model-code formulation ("DeepSeek Sparse Attention", In the code:
    # the top-k set turned into an additive mask over dense attention)
    H, D, Dv, n = 4, 64, 48, 90
    q = rng.standard_normal((H, D)); rows = rng.standard_normal((n, D))
    sel = np.sort(rng.choice(n, size=23, replace=False))
    mask = np.full(n, -np.inf); mask[sel] = 0.0
    o, _ = oracle.sparse_mla(q, rows[sel], 0.125, Dv)
    np.testing.assert_allclose(o, _sdpa_f64(q, rows, 0.125, Dv, mask), rtol=1e-12, atol=1e-12)


def test_mla_closed_forms():
    H, D, Dv = 3, 16, 8
    rows = rng.standard_normal((10, D))
    # Q = 0: uniform weights -> mean of the value dims (the FIRST Dv dims); LSE = log m
    o, lse = oracle.sparse_mla(np.zeros((H, D)), rows, 0.5, Dv)
    for h in range(H):
        np.testing.assert_allclose(o[h], rows[:, :Dv].mean(0), rtol=1e-12)
    np.testing.assert_allclose(lse, np.log(10.0))
    # one selected row: output is its value, LSE is its logit
    q = rng.standard_normal((H, D))
    o, lse = oracle.sparse_mla(q, rows[4:5], 0.5, Dv)
    np.testing.assert_allclose(o, np.repeat(rows[4:5, :Dv], H, 0), rtol=1e-12)
    # two rows along unit directions: weights e^{s*x1} : e^{s*x2} (pins the scale)
    r = np.zeros((2, D)); r[0, 0] = 1.0; r[1, 1] = 1.0; r[0, D - 1] = 5.0; r[1, D - 1] = -5.0
    qq = np.zeros((1, D)); qq[0, 0] = 3.0; qq[0, 1] = 1.0
    scale = 0.7
    o, lse = oracle.sparse_mla(qq, r, scale, D)
    a, b = math.exp(scale * 3.0), math.exp(scale * 1.0)
    np.testing.assert_allclose(o[0], (a * r[0] + b * r[1]) / (a + b), rtol=1e-12)
    np.testing.assert_allclose(lse[0], math.log(a + b), rtol=1e-12)


def test_mla_invariants():
    H, D, Dv = 5, 32, 24
    q = rng.standard_normal((H, D)); rows = rng.standard_normal((17, D))
    o, lse = oracle.sparse_mla(q, rows, 0.3, Dv)
    perm = rng.permutation(17)
    o2, lse2 = oracle.sparse_mla(q, rows[perm], 0.3, Dv)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=1e-12)
    lo = rows[:, :Dv].min(0); hi = rows[:, :Dv].max(0)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)    # convex combination
    same = np.repeat(rows[:1], 6, 0)
    o3, _ = oracle.sparse_mla(q, same, 0.3, Dv)
    np.testing.assert_allclose(o3, np.repeat(rows[:1, :Dv], H, 0), rtol=1e-12)
    o4, lse4 = oracle.sparse_mla(q, rows[:0], 0.3, Dv)
    assert np.all(o4 == 0) and np.all(np.isneginf(lse4))


# ----------------------------------------------------------- whole forward ---

def test_forward_tiny_dense_when_context_within_k():
    spec = W.SPECS["tiny"].scaled(ctx_len=60, q_per_seq=4)       # n <= 64 = k for every query
    wl = W.make_workload(spec)
    res = oracle.dsa_forward(wl)
    assert res.indexer_calls == 0
    seq, pos = wl.query_positions()
    for t in range(wl.total_q):
        np.testing.assert_array_equal(res.idx[t], np.arange(pos[t] + 1))
        # equals dense causal attention computed by the library routine
        rows = oracle.bf16_to_f64(wl.kv[0][: pos[t] + 1])
        ref = _sdpa_f64(oracle.bf16_to_f64(wl.q[0][t]), rows, spec.scale, spec.d_v)
        np.testing.assert_allclose(res.out[0][t], ref, rtol=1e-11, atol=1e-13)


def test_forward_causality_excludes_future_and_includes_self():
    wl = W.make_workload(W.SPECS["tiny"])
    res = oracle.dsa_forward(wl, keep_scores=True)
    seq, pos = wl.query_positions()
    for t in range(wl.total_q):
        assert res.scores[t].shape == (pos[t] + 1,)             # s = 0..p_t
        _check_topk_property(res.scores[t], 64, res.idx[t])
        assert res.idx[t].max() <= pos[t]


def test_indexshare_scores_once_for_the_group():
    # "How GLM5.3 ...", IndexShare: one indexer for 4 layers -> 75% fewer
    # indexer evaluations; every layer attends over the same index set
    spec = W.SPECS["indexshare"].scaled(ctx_len=3000, topk=256, heads=4, d_qk=80, d_v=64, idx_heads=4,
                                        idx_dim=32, batch=2)
    wl = W.make_workload(spec)
    res = oracle.dsa_forward(wl)
    assert res.indexer_calls == wl.total_q                        # not 4 x
    for layer in range(4):
        for t in range(wl.total_q):
            o, l = oracle.attention_on_set(wl, t, layer, res.idx[t])
            np.testing.assert_array_equal(o, res.out[layer][t])
    # per layer, indexer work is 1/4 of one-indexer-per-layer: the page's -75%
    assert 1 - res.indexer_calls / (4 * wl.total_q) == pytest.approx(0.75)


def test_paged_layout_same_as_contiguous():
    spec = W.SPECS["ragged"].scaled(batch=3, ctx_range=(100, 700), topk=128, heads=4, d_qk=80, d_v=64,
                                    idx_heads=4, idx_dim=32)
    wl = W.make_workload(spec)
    # rebuild the same token content in a contiguous pool
    seq, pos = wl.query_positions()
    lens = wl.seq_lens.tolist()
    start = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    rows = np.concatenate([W.pool_rows(wl, b, torch.arange(L)).numpy() for b, L in enumerate(lens)])
    r = torch.from_numpy(rows)
    contig = W.Workload(spec=spec.scaled(paged=False), seq_lens=wl.seq_lens, cu_seqlens_q=wl.cu_seqlens_q,
                        q_idx=wl.q_idx, w=wl.w, k_idx=wl.k_idx[r], q=wl.q, kv=[wl.kv[0][r]],
                        seq_start=torch.from_numpy(start))
    a = oracle.dsa_forward(wl); b = oracle.dsa_forward(contig)
    for t in range(wl.total_q):
        np.testing.assert_array_equal(a.idx[t], b.idx[t])
        np.testing.assert_array_equal(a.out[0][t], b.out[0][t])


def test_band_check_accepts_exact_and_rejects_wrong():
    s = rng.standard_normal(500)
    sel = oracle.topk_select(s, 50)
    assert oracle.band_check(s, 50, sel)[0] == []
    bad = sel.copy(); bad[0] = int(np.argmin(s))
    assert oracle.band_check(s, 50, np.sort(bad))[0] != []


# ------------------------------------------------------ printed figures -----

def test_page_figures_golden():
    with open(os.path.join(GOLDEN, "page_figures.json")) as f:
        g = json.load(f)
    # 64 query heads, 576-d latent with 512-d values: decode intensity vs the
    # page's 120.8 FLOP/B
    got = accounting.decode_intensity(g["query_heads"]["value"], 576, 512)
    assert got == pytest.approx(g["decode_intensity_flop_per_byte"]["value"], rel=1e-3)
    assert W.SPECS["decode"].topk == g["index_topk"]["value"]
    assert W.SPECS["indexshare"].n_layers == g["indexshare_group"]["value"]
    assert W.SPECS["decode"].idx_heads == g["index_n_heads"]["value"]
    assert W.SPECS["decode"].idx_dim == g["index_head_dim"]["value"]


def test_tiny_golden_indices():
    # regression pin: written by tests/golden/make_golden.py from the oracle
    with open(os.path.join(GOLDEN, "tiny_topk.json")) as f:
        g = json.load(f)
    wl = W.make_workload(W.SPECS["tiny"])
    res = oracle.dsa_forward(wl)
    for t, row in enumerate(g["idx"]):
        assert res.idx[t].tolist() == row


def test_workload_recipe():
    wl = W.make_workload(W.SPECS["tiny"])
    seq, pos = wl.query_positions()
    assert pos == list(range(496, 512))
    again = W.make_workload(W.SPECS["tiny"])
    assert torch.equal(wl.k_idx, again.k_idx) and torch.equal(wl.kv[0], again.kv[0])
    assert set(torch.unique(wl.w).tolist()) <= {0.5, 1.0, 2.0}
    assert int(wl.q_idx.float().abs().max()) <= 3
    sp = W.SPECS["ragged"].scaled(batch=5, ctx_range=(100, 300))
    wr = W.make_workload(sp)
    allrows = torch.cat([W.pool_rows(wr, b, torch.arange(int(L))) for b, L in enumerate(wr.seq_lens.tolist())])
    assert torch.unique(allrows).numel() == allrows.numel()       # pages never overlap


# ------------------------------------------------------------ cache append ---

def _tiny_paged_workload():
    # two sequences of 70 and 130 tokens, one query each (their last tokens),
    # 64-token pages: sequence 0 on physical pages (2, 0), sequence 1 on (1, 3, 4)
    spec = W.SPECS["ragged"].scaled(batch=2, ctx_range=(70, 130), topk=16, heads=2, d_qk=80, d_v=64,
                                    idx_heads=4, idx_dim=32)
    g = torch.Generator().manual_seed(5)
    rows = 5 * 64
    return W.Workload(spec=spec, seq_lens=torch.tensor([70, 130], dtype=torch.int32),
                      cu_seqlens_q=torch.tensor([0, 1, 2], dtype=torch.int32),
                      q_idx=torch.zeros((2, 4, 32), dtype=torch.bfloat16), w=torch.ones((2, 4)),
                      k_idx=torch.randn((rows, 32), generator=g).to(torch.bfloat16),
                      q=[torch.zeros((2, 2, 80), dtype=torch.bfloat16)],
                      kv=[torch.randn((rows, 80), generator=g).to(torch.bfloat16)],
                      page_table=torch.tensor([[2, 0, -1], [1, 3, 4]], dtype=torch.int32))


def test_cache_append_hand_computed_rows():
    # token 69 of sequence 0: page 1 -> physical 0, offset 5 -> row 5;
    # token 129 of sequence 1: page 2 -> physical 4, offset 1 -> row 257
    wl = _tiny_paged_workload()
    new = torch.arange(2 * 32, dtype=torch.float32).reshape(2, 32).to(torch.bfloat16) + 1
    out = oracle.cache_append(wl, wl.k_idx, new)
    assert torch.equal(out[5], new[0]) and torch.equal(out[257], new[1])
    keep = torch.ones(out.shape[0], dtype=torch.bool)
    keep[[5, 257]] = False
    assert torch.equal(out[keep], wl.k_idx[keep])


@pytest.mark.parametrize("name,kw", [("decode", dict(ctx_len=700)), ("ragged", dict(ctx_range=(300, 900))),
                                     ("prefill", dict(ctx_len=700, q_per_seq=9))])
def test_cache_append_restores_the_generated_cache(name, kw):
    # the workload generator placed every token's row; blanking the query
    # tokens' rows and appending them again must give the generated pool back,
    # and the forward must not change
    spec = W.SPECS[name].scaled(batch=3, topk=128, heads=4, d_qk=80, d_v=64, idx_heads=4, idx_dim=32, **kw)
    wl = W.make_workload(spec)
    seq, pos = wl.query_positions()
    at = torch.cat([W.pool_rows(wl, b, torch.tensor([p])) for b, p in zip(seq, pos)])
    new_k, new_c = wl.k_idx[at].clone(), wl.kv[0][at].clone()
    blank_k, blank_c = wl.k_idx.clone(), wl.kv[0].clone()
    blank_k[at] = 0
    blank_c[at] = 0
    got_k = oracle.cache_append(wl, blank_k, new_k)
    got_c = oracle.cache_append(wl, blank_c, new_c)
    assert torch.equal(got_k, wl.k_idx) and torch.equal(got_c, wl.kv[0])
    import dataclasses
    again = dataclasses.replace(wl, k_idx=got_k, kv=[got_c])
    a, b = oracle.dsa_forward(wl), oracle.dsa_forward(again)
    for t in range(wl.total_q):
        np.testing.assert_array_equal(a.idx[t], b.idx[t])
        np.testing.assert_array_equal(a.out[0][t], b.out[0][t])


# ------------------------------------------------------ compressed entries ---

def test_compressed_entries_visible_by_brute_force():
    # an entry is visible once every token of its block is at or before the
    # query: enumerate blocks and tokens instead of using the floor formula
    for ratio in (1, 2, 3, 4, 7):
        for p in range(0, 40):
            seen = 0
            for j in range(0, 100):
                if all(tok <= p for tok in range(ratio * j, ratio * j + ratio)):
                    seen += 1
            assert oracle.visible_entries(p, ratio) == seen


def test_compressed_forward_equals_token_forward_on_the_same_rows():
    # a cache of m-token entries whose entry j holds token j's row of an
    # uncompressed cache: a query at token position m (p + 1) - 1 sees p + 1
    # entries, exactly tokens 0..p of the uncompressed cache, so its selection
    # and attention must equal the uncompressed query at position p
    import dataclasses
    m = 3
    spec1 = W.SPECS["tiny"].scaled(ctx_len=300, q_per_seq=5, topk=64)
    w1 = W.make_workload(spec1)
    seq, pos = w1.query_positions()
    specm = spec1.scaled(compress_ratio=m, ctx_len=m * 300)
    wm = dataclasses.replace(w1, spec=specm, seq_lens=w1.seq_lens * m,
                             cu_seqlens_q=w1.cu_seqlens_q)
    # query i of wm sits at token position m*300 - 5 + i; shift the queries so
    # that each lands at m (p + 1) - 1: rebuild with one query per sequence
    a = oracle.dsa_forward(w1)
    for t in range(w1.total_q):
        p = pos[t]
        wq = dataclasses.replace(wm, seq_lens=torch.tensor([m * (p + 1)], dtype=torch.int32),
                                 cu_seqlens_q=torch.tensor([0, 1], dtype=torch.int32),
                                 q_idx=w1.q_idx[t:t + 1], w=w1.w[t:t + 1], q=[w1.q[0][t:t + 1]])
        bq = oracle.dsa_forward(wq)
        np.testing.assert_array_equal(bq.idx[0], a.idx[t])
        np.testing.assert_array_equal(bq.out[0][0], a.out[0][t])
        np.testing.assert_array_equal(bq.lse[0][0], a.lse[0][t])


def test_compressed_dense_when_entries_fit_top_k():
    # k >= visible entries: every entry is attended, i.e. dense attention over
    # the entries (torch's SDPA in float64)
    spec = W.SPECS["tiny"].scaled(ctx_len=4 * 50, q_per_seq=3, topk=64, compress_ratio=4)
    wl = W.make_workload(spec)
    res = oracle.dsa_forward(wl)
    assert res.indexer_calls == 0
    seq, pos = wl.query_positions()
    for t in range(wl.total_q):
        n = (pos[t] + 1) // 4
        np.testing.assert_array_equal(res.idx[t], np.arange(n))
        rows = oracle.bf16_to_f64(wl.kv[0][:n])
        ref = _sdpa_f64(oracle.bf16_to_f64(wl.q[0][t]), rows, spec.scale, spec.d_v)
        np.testing.assert_allclose(res.out[0][t], ref, rtol=1e-11, atol=1e-13)


def test_compressed_workload_layout():
    for name in ("csa_flash", "csa_pro"):
        spec = W.SPECS[name].scaled(batch=3, ctx_len=4000)
        wl = W.make_workload(spec)
        assert wl.k_idx.shape[0] == 3 * (4000 // spec.compress_ratio)
        assert spec.topk in (512, 1024) and spec.idx_heads == 64 and spec.idx_dim == 128
    ps = W.SPECS["csa_flash"].scaled(batch=4, ctx_len=None, ctx_range=(300, 5000), paged=True)
    wp = W.make_workload(ps)
    allrows = torch.cat([W.pool_rows(wp, b, torch.arange(int(L) // 4)) for b, L in enumerate(wp.seq_lens.tolist())])
    assert torch.unique(allrows).numel() == allrows.numel()


# ------------------------------------------------------- HiSparse LRU cache ---

def test_lru_hand_worked_trace():
    with open(os.path.join(GOLDEN, "lru_trace.json")) as f:
        g = json.load(f)
    c = oracle.HiSparseLRU(g["capacity"])
    for st in g["steps"]:
        hits, misses, evicted = c.step(st["request"])
        assert hits == st["hits"] and misses == st["misses"] and evicted == st["evicted"], st
        assert list(c.order) == st["order_after"], st


def test_lru_closed_forms():
    r = np.random.default_rng(3)
    # capacity >= every row ever requested: nothing is evicted, a request hits
    # exactly when the row was requested before
    c = oracle.HiSparseLRU(1000)
    seen = set()
    for _ in range(30):
        req = r.choice(200, size=40, replace=False).tolist()
        hits, misses, evicted = c.step(req)
        assert evicted == [] and set(hits) == set(req) & seen and set(misses) == set(req) - seen
        seen |= set(req)
    # capacity = request size and disjoint requests: every step misses
    # everything and evicts the whole previous step
    c = oracle.HiSparseLRU(50)
    prev = []
    for s in range(6):
        req = list(range(50 * s, 50 * s + 50))
        hits, misses, evicted = c.step(req)
        assert hits == [] and misses == req and sorted(evicted) == sorted(prev)
        prev = req


def test_lru_invariants_on_random_traces():
    r = np.random.default_rng(4)
    for cap in (16, 40, 100):
        c = oracle.HiSparseLRU(cap)
        last_use = {}
        for s in range(60):
            req = r.choice(150, size=int(r.integers(1, 16)), replace=True).tolist()
            before = set(c.order)
            hits, misses, evicted = c.step(req)
            want = set(req)
            assert want <= set(c.order) and len(c.order) <= cap
            assert set(hits) == want & before and set(misses) == want - before
            assert not (set(evicted) & want)
            # no evicted row was used more recently than a kept row that this
            # step did not request
            kept_old = set(c.order) - want
            if evicted and kept_old:
                assert max(last_use[e] for e in evicted) <= min(last_use[k] for k in kept_old)
            for x in want:
                last_use[x] = s


# --------------------------------------------------------------- MHA mode ---

def test_mha_hand_computed_example():
    # one head, latent L = 2 plus one rope dim, one no-rope key dim, one value dim
    c = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, -1.0]])
    w_uk = np.array([[[1.0, 2.0]]])            # k_nope(s) = c0 + 2 c1
    w_uv = np.array([[[3.0, -1.0]]])           # v(s) = 3 c0 - c1
    K, V = oracle.mha_upproject(c, w_uk, w_uv)
    np.testing.assert_array_equal(K[:, 0, :], [[1.0, 2.0], [2.0, -1.0]])
    np.testing.assert_array_equal(V[:, 0, :], [[3.0], [-1.0]])
    O, lse = oracle.sparse_mha(np.array([[1.0, 1.0]]), K, V, 1.0)
    p0 = 1.0 / (1.0 + math.exp(-2.0))          # logits 3 and 1
    assert abs(O[0, 0] - (4.0 * p0 - 1.0)) < 1e-15
    assert abs(lse[0] - (3.0 + math.log1p(math.exp(-2.0)))) < 1e-15


def test_mha_equals_mqa_with_absorbed_projections():
    # q_nope . (W_UK c) = (W_UK^T q_nope) . c and sum p (W_UV c) = W_UV sum p c: MHA mode
    # is the MQA latent attention with the absorbed query, its output up-projected
    rng = np.random.default_rng(7)
    H, L, rope, dn, dv, m = 3, 16, 4, 6, 5, 9
    c = rng.normal(size=(m, L + rope))
    w_uk = rng.normal(size=(H, dn, L))
    w_uv = rng.normal(size=(H, dv, L))
    q = rng.normal(size=(H, dn + rope))
    scale = 0.3
    K, V = oracle.mha_upproject(c, w_uk, w_uv)
    O, lse = oracle.sparse_mha(q, K, V, scale)
    q_abs = np.stack([np.concatenate([w_uk[h].T @ q[h, :dn], q[h, dn:]]) for h in range(H)])
    o_lat, lse_lat = oracle.sparse_mla(q_abs, c, scale, L)
    for h in range(H):
        np.testing.assert_allclose(O[h], w_uv[h] @ o_lat[h], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_lat, rtol=1e-12, atol=1e-12)


def test_mha_dense_case_equals_library_attention():
    rng = np.random.default_rng(3)
    H, m, dqk, dv = 4, 13, 8, 6
    K = rng.normal(size=(m, H, dqk))
    V = rng.normal(size=(m, H, dv))
    q = rng.normal(size=(H, dqk))
    O, lse = oracle.sparse_mha(q, K, V, 0.5)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], torch.from_numpy(K).permute(1, 0, 2), torch.from_numpy(V).permute(1, 0, 2),
        scale=0.5)
    np.testing.assert_allclose(O, ref[:, 0, :].numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(0.5 * torch.einsum("hd,mhd->hm", torch.from_numpy(q), torch.from_numpy(K)), dim=1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_mha_order_invariant_and_empty_selection():
    rng = np.random.default_rng(5)
    K = rng.normal(size=(7, 2, 4))
    V = rng.normal(size=(7, 2, 3))
    q = rng.normal(size=(2, 4))
    perm = rng.permutation(7)
    a = oracle.sparse_mha(q, K, V, 1.0)
    b = oracle.sparse_mha(q, K[perm], V[perm], 1.0)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-13)
    O, lse = oracle.sparse_mha(q, K[:0], V[:0], 1.0)
    assert (O == 0).all() and np.isneginf(lse).all()


def test_mha_workload_reads_the_selected_rows():
    spec = W.SPECS["mha"].scaled(ctx_len=300, q_per_seq=20, idx_heads=4, idx_dim=32, topk=64, heads=2)
    wl = W.make_workload(spec)
    seq, pos = wl.query_positions()
    t = 5
    sel = np.array([3, 40, -1, 17], dtype=np.int64)
    O, lse = oracle.mha_attention_on_set(wl, t, 0, sel)
    rows = W.pool_rows(wl, seq[t], torch.tensor([3, 40, 17]))
    c = oracle.bf16_to_f64(wl.kv[0][rows])
    K, V = oracle.mha_upproject(c, oracle.bf16_to_f64(wl.w_uk[0]), oracle.bf16_to_f64(wl.w_uv[0]))
    O2, lse2 = oracle.sparse_mha(oracle.bf16_to_f64(wl.q_mha[0][t]), K, V, spec.scale)
    np.testing.assert_array_equal(O, O2)
    assert wl.q_mha[0].shape == (20, 2, 256) and wl.w_uk[0].shape == (2, 192, 512)
    assert wl.w_uv[0].shape == (2, 256, 512)
    assert pos[0] == 280 and pos[-1] == 299
