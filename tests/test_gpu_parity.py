"""Parity of the CUDA path (through the C ABI) with the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import check_output, compare_forward, make_sa, sel_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


# ------------------------------------------------ device machinery checks ---

@pytest.mark.parametrize("a_mn,b_mn,sw", [(False, False, 128), (True, True, 128), (True, False, 128),
                                          (False, True, 128), (False, False, 64),
                                          (False, False, 0), (False, True, 0)])  # 0: A from tensor memory
def test_selftest_mma_tile(lib, a_mn, b_mn, sw):
    g = torch.Generator().manual_seed(7)
    a = torch.randint(-4, 5, (128, 64), generator=g).to(torch.bfloat16).cuda()
    b = torch.randint(-4, 5, (64, 64), generator=g).to(torch.bfloat16).cuda()
    d = torch.zeros((128, 64), dtype=torch.float32, device="cuda")
    lib.selftest_mma(a, b, d, a_mn, b_mn, sw)
    assert lib.check_device_error() == lib.DSA_OK
    ref = a.double().cpu() @ b.double().cpu().T
    assert torch.equal(d.cpu().double(), ref), f"tile mismatch (a_mn={a_mn}, b_mn={b_mn}, swizzle {sw})"


def test_bounded_wait_reports_timeout(lib):
    lib.selftest_timeout(50)
    assert lib.check_device_error() == lib.DSA_ERR_TIMEOUT
    assert lib.check_device_error() == lib.DSA_OK        # the word was cleared
    x = torch.ones(4, device="cuda") * 2                 # context still usable
    assert float(x.sum()) == 8.0


# -------------------------------------------------------- tiny: bit exact ---

def test_tiny_forward_exact(lib):
    wl = W.make_workload(W.SPECS["tiny"]).to("cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q), exact_idx=True)


def test_tiny_indexer_scores_exact(lib):
    wl = W.make_workload(W.SPECS["tiny"]).to("cuda")
    sa = make_sa(wl)
    T, L = wl.total_q, wl.max_seqlen_k
    scores = torch.full((T, L), float("nan"), dtype=torch.float32, device="cuda")
    lib.indexer_scores(sa.batch, sa.indexer, scores, sa.workspace, skip_dense_k=0)
    assert lib.check_device_error() == lib.DSA_OK
    got = scores.cpu().numpy()
    cpu = wl.to("cpu")
    seq, pos = cpu.query_positions()
    for t in range(T):
        ref = oracle.scores_for_query(cpu, t)
        assert np.array_equal(got[t, : pos[t] + 1].astype(np.float64), ref), f"query {t}"
        assert np.all(np.isnan(got[t, pos[t] + 1:])), "entries past the causal context must stay unwritten"


@pytest.mark.parametrize("n,k,kind,cap", [
    (5000, 2048, "normal", 0), (3000, 2048, "ties", 0), (40000, 2048, "normal", 0), (2000, 2048, "normal", 0),
    (700, 64, "zeros", 0), (1048576, 2048, "normal", 0),
    # ties at the k-th key spread over the blocks of 16-block clusters
    (200000, 2048, "ties2", 0), (1048576, 2048, "ties2", 0), (1048576, 2048, "ties_top", 0),
    # clusters capped at 8 blocks: 131072 keys per block, 128-key runs per thread
    # (the write path that re-reads its run instead of keeping bitmasks)
    (1048576, 2048, "ties2", 8), (1048576, 2048, "normal", 8), (300000, 1000, "ties_top", 2)])
def test_topk_exact_on_given_scores(lib, n, k, kind, cap):
    # both sides decide on the same fp32 values: the selection must match bit for bit
    g = torch.Generator().manual_seed(n + k)
    T = 3
    if kind == "normal":
        s = torch.randn((T, n), generator=g)
    elif kind == "ties":
        s = torch.randint(-5, 6, (T, n), generator=g).float()
    elif kind == "ties2":
        s = torch.randint(-2, 3, (T, n), generator=g).float()
    elif kind == "ties_top":
        # a few hundred keys above a huge run of equal keys spread over the whole
        # row: the equal keys taken must be the lowest positions, whichever block holds them
        s = torch.zeros((T, n))
        s[:, torch.randperm(n, generator=g)[:300]] = 1.0
    else:  # signed zeros and a few positives
        s = torch.zeros((T, n))
        s[:, ::3] = -0.0
        s[:, 7::97] = 1.0
    ld = (n + 3) // 4 * 4
    scores = torch.zeros((T, ld), dtype=torch.float32)
    scores[:, :n] = s
    scores = scores.cuda()
    cu = torch.arange(T + 1, dtype=torch.int32, device="cuda")
    lens = torch.full((T,), n, dtype=torch.int32, device="cuda")
    batch = lib.make_batch(cu, lens, T, n, 1)
    ws = torch.empty(lib.workspace_size(batch, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    lib.selftest_topk_max_cluster(cap)
    try:
        lib.topk(batch, scores, k, idx, ws)
        assert lib.check_device_error() == lib.DSA_OK
    finally:
        lib.selftest_topk_max_cluster(0)
    got = idx.cpu().numpy()
    for t in range(T):
        ref = oracle.topk_select(s[t].double().numpy(), k)
        sel = sel_of(got[t])
        assert np.array_equal(sel, ref), f"row {t}"
        assert np.all(got[t][len(sel):] == -1)


def test_sparse_mla_on_oracle_indices(lib):
    # decode shapes, a few queries, index sets chosen by the oracle, plus -1 holes
    spec = W.SPECS["decode"].scaled(batch=3, ctx_len=9000)
    wl = W.make_workload(spec, device="cuda")
    cpu = wl.to("cpu")
    ref = oracle.dsa_forward(cpu)
    T, k = wl.total_q, spec.topk
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for t in range(T):
        sel = ref.idx[t].copy()
        sel[::17] = -1                      # holes are skipped
        idx[t, : len(sel)] = torch.from_numpy(sel.astype(np.int32))
    idx = idx.cuda()
    sa = make_sa(wl)
    out = torch.empty((T, spec.heads, spec.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, spec.heads), dtype=torch.float32, device="cuda")
    lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx, k, out, lse, sa.workspace)
    assert lib.check_device_error() == lib.DSA_OK
    for t in range(T):
        o, l = oracle.attention_on_set(cpu, t, 0, idx[t].cpu().numpy())
        check_output(out[t].float().cpu().numpy(), o, f"query {t}")
        np.testing.assert_allclose(lse[t].cpu().numpy(), l, rtol=1e-4, atol=1e-4)


# ------------------------------------------------- workloads, smaller sizes ---

@pytest.mark.parametrize("ctx", [2047, 2048, 2049, 4100, 9000])
def test_decode_small_contexts(lib, ctx):
    # around the dense threshold (n <= k selects everything) and ragged tails
    spec = W.SPECS["decode"].scaled(batch=4, ctx_len=ctx)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))


def test_prefill_small_chunk(lib):
    spec = W.SPECS["prefill"].scaled(ctx_len=6000, q_per_seq=70)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, [0, 1, 2, 33, 68, 69])


def test_ragged_paged_small(lib):
    spec = W.SPECS["ragged"].scaled(batch=9, ctx_range=(100, 5000))
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))


def test_indexshare_small(lib):
    spec = W.SPECS["indexshare"].scaled(ctx_len=20000)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))


# ------------------------------------------------------------- invariants ---

def test_paged_equals_contiguous_bitwise(lib):
    spec = W.SPECS["ragged"].scaled(batch=6, ctx_range=(1500, 6000))
    wl = W.make_workload(spec, device="cuda")
    lens = wl.seq_lens.tolist()
    rows = torch.cat([W.pool_rows(wl, b, torch.arange(L)) for b, L in enumerate(lens)]).cuda()
    start = torch.zeros(len(lens), dtype=torch.int64)
    start[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)[:-1]
    contig = W.Workload(spec=spec.scaled(paged=False), seq_lens=wl.seq_lens, cu_seqlens_q=wl.cu_seqlens_q,
                        q_idx=wl.q_idx, w=wl.w, k_idx=wl.k_idx[rows].contiguous(), q=wl.q,
                        kv=[wl.kv[0][rows].contiguous()], seq_start=start.cuda())
    a_idx, a_out, _ = make_sa(wl).forward()
    b_idx, b_out, _ = make_sa(contig).forward()
    assert lib.check_device_error() == lib.DSA_OK
    assert torch.equal(a_idx, b_idx)
    assert torch.equal(a_out[0], b_out[0])


def test_batched_equals_alone_bitwise(lib):
    spec = W.SPECS["decode"].scaled(batch=5, ctx_len=7000)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, _ = make_sa(wl).forward()
    one = W.Workload(spec=spec.scaled(batch=1), seq_lens=wl.seq_lens[2:3], cu_seqlens_q=wl.cu_seqlens_q[:2],
                     q_idx=wl.q_idx[2:3], w=wl.w[2:3], k_idx=wl.k_idx, q=[wl.q[0][2:3]], kv=wl.kv,
                     seq_start=wl.seq_start[2:3])
    i1, o1, _ = make_sa(one).forward()
    assert lib.check_device_error() == lib.DSA_OK
    assert torch.equal(idx[2], i1[0])
    assert torch.equal(outs[0][2], o1[0][0])


def test_indexshare_layers_read_one_index_set(lib):
    spec = W.SPECS["indexshare"].scaled(ctx_len=9000)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx, outs, _ = sa.forward()
    # the same layer run alone on that index set reproduces each layer bitwise
    for layer in range(4):
        out = torch.empty_like(outs[layer])
        from long_context_lightning_gb300 import _lib
        _lib.sparse_mla_fwd(sa.batch, sa.layers[layer], idx, spec.topk, out, None, sa.workspace)
        assert torch.equal(out, outs[layer]), f"layer {layer}"
    assert lib.check_device_error() == lib.DSA_OK


def test_bad_index_is_flagged_not_trapped(lib):
    spec = W.SPECS["decode"].scaled(batch=2, ctx_len=3000)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx = torch.arange(spec.topk, dtype=torch.int32, device="cuda").repeat(2, 1)
    idx[1, 5] = 999999                         # beyond the causal context
    out = torch.empty((2, spec.heads, spec.d_v), dtype=torch.bfloat16, device="cuda")
    lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx, spec.topk, out, None, sa.workspace)
    assert lib.check_device_error() == lib.DSA_ERR_BAD_INDEX
    # the row is still computed over the remaining valid positions
    cpu = wl.to("cpu")
    o, _ = oracle.attention_on_set(cpu, 1, 0, np.delete(np.arange(spec.topk), 5))
    check_output(out[1].float().cpu().numpy(), o, "row with a bad index")


def test_host_validation(lib):
    spec = W.SPECS["tiny"]
    wl = W.make_workload(spec).to("cuda")
    sa = make_sa(wl)
    bad = torch.empty((wl.total_q, 4096), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.DsaError) as e:
        lib.topk(sa.batch, sa.scores_view(), 4096, bad, sa.workspace)   # k > 2048
    assert e.value.status == lib.DSA_ERR_UNSUPPORTED
    tiny_ws = sa.workspace[:16]
    with pytest.raises(lib.DsaError) as e:
        lib.forward(sa.batch, sa.indexer, spec.topk, sa.layers, sa.idx, sa.outs, None, tiny_ws)
    assert e.value.status == lib.DSA_ERR_WORKSPACE


def test_empty_selection_row(lib):
    spec = W.SPECS["decode"].scaled(batch=1, ctx_len=3000)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx = torch.full((1, spec.topk), -1, dtype=torch.int32, device="cuda")
    out = torch.full((1, spec.heads, spec.d_v), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, spec.heads), dtype=torch.float32, device="cuda")
    lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx, spec.topk, out, lse, sa.workspace)
    assert lib.check_device_error() == lib.DSA_OK
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("n,k,kind,cap", [
    (32768, 2048, "normal", 0), (32768, 2048, "ties_top", 0), (131072, 2048, "normal", 0),
    (1048576, 2048, "normal", 0), (300000, 2048, "ties", 0), (9000, 2048, "normal", 1),
    (40000, 512, "normal", 0), (200000, 1024, "narrow", 0), (50000, 2048, "narrow", 4)])
def test_topk_candidate_and_three_pass_paths_agree(lib, n, k, kind, cap):
    # the candidate path (first digit across the cluster, the rest in one block)
    # and the three-pass path must both give the oracle's selection
    g = torch.Generator().manual_seed(3 * n + k)
    T = 4
    if kind == "normal":
        s = torch.randn((T, n), generator=g)
    elif kind == "ties":
        s = torch.randint(-40, 41, (T, n), generator=g).float()
    elif kind == "narrow":   # many keys in the threshold's first-digit bin
        s = 1.0 + torch.rand((T, n), generator=g) * 1e-3
    else:
        s = torch.zeros((T, n))
        s[:, torch.randperm(n, generator=g)[:300]] = 1.0
    ld = (n + 3) // 4 * 4
    scores = torch.zeros((T, ld), dtype=torch.float32)
    scores[:, :n] = s
    scores = scores.cuda()
    cu = torch.arange(T + 1, dtype=torch.int32, device="cuda")
    lens = torch.full((T,), n, dtype=torch.int32, device="cuda")
    batch = lib.make_batch(cu, lens, T, n, 1)
    ws = torch.empty(lib.workspace_size(batch, k), dtype=torch.uint8, device="cuda")
    got = {}
    lib.selftest_topk_max_cluster(cap)
    try:
        for cand in (True, False):
            idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
            lib.selftest_topk_path(cand)
            lib.topk(batch, scores, k, idx, ws)
            assert lib.check_device_error() == lib.DSA_OK
            got[cand] = idx.cpu()
    finally:
        lib.selftest_topk_path(True)
        lib.selftest_topk_max_cluster(0)
    assert torch.equal(got[True], got[False])
    for t in range(T):
        ref = oracle.topk_select(s[t].double().numpy(), k)
        assert np.array_equal(sel_of(got[True][t].numpy()), ref), f"row {t}"


@pytest.mark.parametrize("cap", [0, 4])
def test_topk_many_rows_mixed_paths(lib, cap):
    # more rows than clusters fit on the GPU at once: each cluster takes a share
    # of the rows, alternating dense rows, candidate-path rows and rows whose
    # threshold bin is too large for the candidates (three-pass path)
    g = torch.Generator().manual_seed(99 + cap)
    T, k = 700, 512
    lens = torch.randint(100, 40000, (T,), generator=g)
    lens[::7] = torch.randint(10, k + 1, (len(lens[::7]),), generator=g)   # dense rows
    n_max = int(lens.max())
    ld = (n_max + 3) // 4 * 4
    scores = torch.randn((T, ld), generator=g)
    scores[1::5] = 2.0 + torch.rand((len(scores[1::5]), ld), generator=g) * 1e-4  # one huge threshold bin
    scores[2::9] = torch.randint(-3, 4, (len(scores[2::9]), ld), generator=g).float()
    cu = torch.arange(T + 1, dtype=torch.int32).cuda()
    lens_d = lens.to(torch.int32).cuda()
    batch = lib.make_batch(cu, lens_d, T, n_max, 1)
    ws = torch.empty(lib.workspace_size(batch, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    lib.selftest_topk_max_cluster(cap)
    try:
        lib.topk(batch, scores.cuda(), k, idx, ws)
        assert lib.check_device_error() == lib.DSA_OK
    finally:
        lib.selftest_topk_max_cluster(0)
    got = idx.cpu().numpy()
    for t in range(T):
        n = int(lens[t])
        ref = oracle.topk_select(scores[t, :n].double().numpy(), k)
        sel = sel_of(got[t])
        assert np.array_equal(sel, ref), f"row {t} (n={n})"
        assert np.all(got[t][len(sel):] == -1)
