"""The fused forward over compressed cache entries (top-512 / top-1024 entries
of caches holding one entry per 4 tokens), against the float64 oracle: the
entry selection bit-exact on integer-valued indexer inputs, within the tie
band on normal ones, and the attention over the GPU's own selected entries
within the stated tolerances."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import compare_forward, make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


@pytest.mark.parametrize("name", ["csa_flash", "csa_pro"])
def test_compressed_full_size(lib, name):
    spec = W.SPECS[name]
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))


@pytest.mark.parametrize("name", ["csa_flash", "csa_pro"])
def test_compressed_integer_exact(lib, name):
    spec = W.SPECS[name].scaled(integer_indexer=True, batch=8)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx, outs, lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    cpu = wl.to("cpu")
    compare_forward(cpu, idx, outs, lses, range(wl.total_q), exact_idx=True)
    # the fused call's fp32 scores are the oracle's, bit for bit, over every visible entry
    scores = sa.scores_view().double().cpu().numpy()
    seq, pos = cpu.query_positions()
    for t in range(wl.total_q):
        n = oracle.visible_entries(pos[t], spec.compress_ratio)
        assert np.array_equal(scores[t, :n], oracle.scores_for_query(cpu, t)), f"query {t}"


@pytest.mark.parametrize("ratio,ctx", [(4, 8195), (4, 8196), (3, 6145), (7, 40000)])
def test_compressed_around_the_dense_threshold_and_partial_blocks(lib, ratio, ctx):
    # 8195 tokens / 4 -> 2048 entries (dense at k = 2048), 8196 -> 2049 visible
    # for the last query; 3 and 7 tokens per entry leave partial blocks
    spec = W.SPECS["csa_flash"].scaled(batch=3, ctx_len=ctx, q_per_seq=2, topk=2048, compress_ratio=ratio)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))


def test_compressed_paged_equals_contiguous_bitwise(lib):
    spec = W.SPECS["csa_flash"].scaled(batch=5, ctx_len=None, ctx_range=(3000, 20000), paged=True)
    wl = W.make_workload(spec, device="cuda")
    lens = [int(L) // spec.compress_ratio for L in wl.seq_lens.tolist()]
    rows = torch.cat([W.pool_rows(wl, b, torch.arange(L)) for b, L in enumerate(lens)]).cuda()
    start = torch.zeros(len(lens), dtype=torch.int64)
    start[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)[:-1]
    contig = W.Workload(spec=spec.scaled(paged=False), seq_lens=wl.seq_lens, cu_seqlens_q=wl.cu_seqlens_q,
                        q_idx=wl.q_idx, w=wl.w, k_idx=wl.k_idx[rows].contiguous(), q=wl.q,
                        kv=[wl.kv[0][rows].contiguous()], seq_start=start.cuda())
    a_idx, a_out, _ = make_sa(wl).forward()
    b_idx, b_out, _ = make_sa(contig).forward()
    assert lib.check_device_error() == lib.DSA_OK
    assert torch.equal(a_idx, b_idx) and torch.equal(a_out[0], b_out[0])
    compare_forward(wl.to("cpu"), a_idx, a_out, None, range(wl.total_q))
