"""Cache append on the GPU against the float64 oracle's plain per-token writes:
the query tokens' rows of the indexer-key pool and of every latent pool,
paged and contiguous, bit for bit; the forward over the appended caches equals
the forward over the generated ones bit for bit."""
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


@pytest.mark.parametrize("name,kw", [("decode", dict(batch=8, ctx_len=5000)),
                                     ("ragged", dict(batch=16, ctx_range=(100, 9000))),
                                     ("prefill", dict(ctx_len=6000, q_per_seq=70)),
                                     ("indexshare", dict(batch=2, ctx_len=12000))])
def test_append_then_forward_matches_generated_cache(lib, name, kw):
    spec = W.SPECS[name].scaled(**kw)
    wl = W.make_workload(spec, device="cuda")
    sa_ref = make_sa(wl)
    idx_ref, outs_ref, _ = sa_ref.forward()
    torch.cuda.synchronize()
    seq, pos = wl.query_positions()
    at = torch.cat([W.pool_rows(wl, b, torch.tensor([p])) for b, p in zip(seq, pos)]).cuda()
    new_k = wl.k_idx[at].clone()
    new_c = [kv[at].clone() for kv in wl.kv]
    orig_k = wl.k_idx.clone()
    orig_c = [kv.clone() for kv in wl.kv]
    wl.k_idx[at] = 0
    for kv in wl.kv:
        kv[at] = 0
    cpu = wl.to("cpu")
    sa = make_sa(wl)          # descriptors over the same (now blanked) pools
    lib.cache_append(sa.batch, new_k, sa.indexer.k)
    for layer, c in zip(sa.layers, new_c):
        lib.cache_append(sa.batch, c, layer.kv)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    # bit for bit what the oracle writes, and the generated pools again
    assert torch.equal(wl.k_idx.cpu(), oracle.cache_append(cpu, cpu.k_idx, new_k.cpu()))
    for layer in range(spec.n_layers):
        assert torch.equal(wl.kv[layer].cpu(), oracle.cache_append(cpu, cpu.kv[layer], new_c[layer].cpu()))
        assert torch.equal(wl.kv[layer], orig_c[layer])
    assert torch.equal(wl.k_idx, orig_k)
    idx, outs, _ = sa.forward()
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref)
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a, b)


def test_append_bad_page_is_flagged_not_trapped(lib):
    spec = W.SPECS["ragged"].scaled(batch=4, ctx_range=(200, 3000))
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    seq, pos = wl.query_positions()
    b, p = seq[2], pos[2]
    wl.page_table[b, p // 64] = 10 ** 8          # beyond the pool
    before = wl.k_idx.clone()
    rows = torch.ones((wl.total_q, spec.idx_dim), dtype=torch.bfloat16, device="cuda")
    lib.cache_append(sa.batch, rows, sa.indexer.k)
    assert lib.check_device_error() == lib.DSA_ERR_BAD_INDEX
    changed = (wl.k_idx != before).any(dim=1).nonzero().flatten().cpu().tolist()
    assert len(changed) == wl.total_q - 1        # every other token was written


def test_append_skips_a_malformed_sequence(lib):
    # a sequence with fewer cached tokens than queries has no valid positions:
    # its tokens write nothing and are flagged; every other token is written
    spec = W.SPECS["prefill"].scaled(batch=3, ctx_len=3000, q_per_seq=40)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    wl.seq_lens[1] = 39
    before = wl.k_idx.clone()
    rows = torch.ones((wl.total_q, spec.idx_dim), dtype=torch.bfloat16, device="cuda")
    lib.cache_append(sa.batch, rows, sa.indexer.k)
    assert lib.check_device_error() == lib.DSA_ERR_BAD_INDEX
    changed = set((wl.k_idx != before).any(dim=1).nonzero().flatten().cpu().tolist())
    seq, pos = wl.query_positions()
    wanted = set()
    for t in range(wl.total_q):
        if seq[t] != 1:
            wanted |= set(W.pool_rows(wl, seq[t], torch.tensor([pos[t]])).tolist())
    assert changed == wanted


@pytest.mark.parametrize("name,kw", [("decode", dict(batch=8, ctx_len=5000)),
                                     ("indexshare", dict(batch=2, ctx_len=12000)),
                                     ("ragged", dict(batch=16, ctx_range=(100, 9000)))])
def test_overlapped_forward_with_uploads_on_a_second_stream(lib, name, kw):
    # a serving step: the indexer inputs and keys go in on the main stream, the
    # layers' queries and latent rows on a second one that the sparse MLA waits
    # for, and the index set comes back while the MLA runs; eager and replayed
    # from a CUDA graph, the results equal dsa_forward's bit for bit
    spec = W.SPECS[name].scaled(**kw)
    wl = W.make_workload(spec, device="cuda")
    sa_ref = make_sa(wl)
    idx_ref, outs_ref, lses_ref = [x.clone() if torch.is_tensor(x) else [y.clone() for y in x]
                                   for x in sa_ref.forward()]
    seq, pos = wl.query_positions()
    at = torch.cat([W.pool_rows(wl, b, torch.tensor([p])) for b, p in zip(seq, pos)]).cuda()
    host_q = [q.cpu().pin_memory() for q in wl.q]
    host_c = [kv[at].cpu().pin_memory() for kv in wl.kv]
    host_k = wl.k_idx[at].cpu().pin_memory()
    dev_c = [torch.empty_like(c, device="cuda") for c in host_c]
    dev_k = torch.empty_like(host_k, device="cuda")
    for kv in wl.kv:
        kv[at] = 0
    wl.k_idx[at] = 0
    for q in wl.q:
        q.zero_()
    sa = make_sa(wl)
    host_idx = torch.empty(sa.idx.shape, dtype=sa.idx.dtype).pin_memory()
    side = torch.cuda.Stream()
    fork, ready, done, back = (torch.cuda.Event() for _ in range(4))
    done.record()               # the library records it later: create the event now

    def step():
        main = torch.cuda.current_stream()   # under capture, the capturing stream
        fork.record(main)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            for q, h in zip(wl.q, host_q):
                q.copy_(h, non_blocking=True)
            for layer, c, h in zip(sa.layers, dev_c, host_c):
                c.copy_(h, non_blocking=True)
                lib.cache_append(sa.batch, c, layer.kv, stream=side)
            ready.record(side)
        dev_k.copy_(host_k, non_blocking=True)
        lib.cache_append(sa.batch, dev_k, sa.indexer.k)
        sa.forward_overlapped(mla_ready=ready, topk_done=done)
        side.wait_event(done)
        with torch.cuda.stream(side):
            host_idx.copy_(sa.idx, non_blocking=True)
            back.record(side)
        main.wait_event(back)

    def check():
        torch.cuda.synchronize()
        assert lib.check_device_error() == lib.DSA_OK
        assert torch.equal(host_idx, idx_ref.cpu())
        assert torch.equal(sa.idx, idx_ref)
        for a, b in zip(sa.outs, outs_ref):
            assert torch.equal(a, b)
        for a, b in zip(sa.lses, lses_ref):
            assert torch.equal(a, b)

    step()
    check()
    for x in (sa.idx, *sa.outs, *sa.lses, host_idx):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        step()
    for kv in wl.kv:            # the replay must upload and append everything again
        kv[at] = 0
    wl.k_idx[at] = 0
    for q in wl.q:
        q.zero_()
    g.replay()
    check()
