"""HiSparse on the GPU against the oracle's least-recently-used cache
(oracle.HiSparseLRU): over several steps of selections the hits, misses,
evictions and the resident order agree exactly; every slot holds its host row
bit for bit; sparse MLA over the slot pool equals sparse MLA over the pool
bit for bit; a step that asks for more rows than the cache holds changes
nothing and is reported."""
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import check_lse, check_output, make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


def _selection(wl, step, k):
    """Seeded synthetic selection: k distinct positions of each query's causal
    context (all of it when shorter), a few entries -1; queries of one
    sequence share most of their rows."""
    seq, pos = wl.query_positions()
    T = len(seq)
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for t in range(T):
        n = pos[t] + 1
        g = torch.Generator().manual_seed(1000 * step + 17 * seq[t] + (t % 2))
        m = min(n, k)
        idx[t, :m] = torch.randperm(n, generator=g)[:m].to(torch.int32)
        idx[t, 3:m:97] = -1
    return idx


def _oracle_rows(wl_cpu, idx):
    return oracle.requested_rows(wl_cpu, [r.numpy() for r in idx])


def _entry_rows(wl, idx):
    """Pool row of every entry (-1 where the entry is -1 or beyond the context)."""
    seq, pos = wl.query_positions()
    rows = torch.full(idx.shape, -1, dtype=torch.int64)
    for t in range(idx.shape[0]):
        m = min(pos[t] + 1, idx.shape[1])
        sel = idx[t, :m].to(torch.int64)
        ok = sel >= 0
        rows[t, :m][ok] = W.pool_rows(wl, seq[t], sel[ok])
    return rows


def _cache(wl, host, capacity):
    from long_context_lightning_gb300 import HiSparseCache
    return HiSparseCache(host, capacity, seq_start=wl.seq_start, page_table=wl.page_table,
                         page_size=wl.spec.page_size)


def _setup(lib, spec, capacity):
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    host = wl.kv[0].cpu().pin_memory()
    return wl, sa, host, _cache(wl, host, capacity)


@pytest.mark.parametrize("name,kw,slack", [
    ("ragged", dict(batch=6, ctx_range=(300, 9000), q_per_seq=3), 200),
    ("decode", dict(batch=4, ctx_len=6000), 700),
])
def test_lru_steps_match_oracle(lib, name, kw, slack):
    spec = W.SPECS[name].scaled(**kw)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    host = wl.kv[0].cpu().pin_memory()
    wl_cpu = wl.to("cpu", kv_too=False)
    k = spec.topk
    T = wl.total_q
    idx_f, _, _ = sa.forward()                      # step 1: the indexer's own selection
    sels = [idx_f.cpu()] + [_selection(wl, s, k) for s in range(2, 7)]
    # room for the largest step plus some slack: later steps must evict
    per_step = [_oracle_rows(wl_cpu, i) for i in sels]
    capacity = max(len(r) for r in per_step) + slack
    assert len(set().union(*per_step)) > capacity
    hc = _cache(wl, host, capacity)
    lru = oracle.HiSparseLRU(capacity)
    slots = torch.empty((T, k), dtype=torch.int32, device="cuda")
    total_evicted = 0
    for step, idx in enumerate(sels, start=1):
        idx_d = idx.cuda()
        hc.fetch(sa.batch, idx_d, k, slots)
        assert lib.check_device_error() == lib.DSA_OK
        hits, misses, evicted = lru.step(_oracle_rows(wl_cpu, idx))
        total_evicted += len(evicted)
        st = hc.stats()
        assert st == dict(steps=step, requested=len(hits) + len(misses), hits=len(hits), misses=len(misses),
                          evicted=len(evicted), overflow=0), f"step {step}"
        assert hc.resident() == list(lru.order), f"step {step}: LRU order"
        # every selected entry's slot holds its host row, bit for bit
        rows = _entry_rows(wl_cpu, idx)
        s = slots.cpu()
        assert torch.equal(s < 0, rows < 0)
        valid = rows >= 0
        got = hc.slot_pool[s[valid].to(torch.int64).cuda()].cpu()
        assert torch.equal(got, host[rows[valid]])
        # sparse MLA over the slots equals sparse MLA over the pool
        out_a = torch.empty_like(sa.outs[0])
        lse_a = torch.empty_like(sa.lses[0])
        out_b = torch.empty_like(sa.outs[0])
        lse_b = torch.empty_like(sa.lses[0])
        lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx_d, k, out_a, lse_a, sa.workspace)
        lib.sparse_mla_fwd(sa.batch, hc.layer(wl.q[0], spec.d_v, spec.scale), slots, k, out_b, lse_b,
                           sa.workspace)
        torch.cuda.synchronize()
        assert lib.check_device_error() == lib.DSA_OK
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), f"step {step}"
    assert total_evicted > 0                         # the trace exercised eviction


def test_attention_over_slots_matches_oracle(lib):
    spec = W.SPECS["ragged"].scaled(batch=3, ctx_range=(500, 4000), q_per_seq=2)
    wl, sa, host, hc = _setup(lib, spec, 9000)
    k, T = spec.topk, wl.total_q
    slots = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = torch.empty_like(sa.outs[0])
    lse = torch.empty_like(sa.lses[0])
    idx = _selection(wl, 3, k)
    hc.fetch(sa.batch, idx.cuda(), k, slots)
    lib.sparse_mla_fwd(sa.batch, hc.layer(wl.q[0], spec.d_v, spec.scale), slots, k, out, lse, sa.workspace)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    wl_cpu = wl.to("cpu")
    seq, pos = wl.query_positions()
    for t in range(T):
        sel = idx[t, :min(pos[t] + 1, k)].numpy()
        ref_o, ref_l = oracle.attention_on_set(wl_cpu, t, 0, sel)
        check_output(out[t].float().cpu().numpy(), ref_o, f"query {t}")
        check_lse(lse[t].cpu().numpy(), ref_l, f"query {t}")


def test_capacity_overflow_changes_nothing(lib):
    spec = W.SPECS["decode"].scaled(batch=3, ctx_len=5000)
    wl, sa, host, hc = _setup(lib, spec, 5000)
    wl_cpu = wl.to("cpu", kv_too=False)
    k, T = spec.topk, wl.total_q
    slots = torch.empty((T, k), dtype=torch.int32, device="cuda")
    first = _selection(wl, 2, k)
    first[1:] = -1                                   # one query: 2048 - a few rows, fits
    hc.fetch(sa.batch, first.cuda(), k, slots)
    assert lib.check_device_error() == lib.DSA_OK
    before = hc.resident()
    want = _oracle_rows(wl_cpu, _selection(wl, 5, k))
    assert len(want) > 5000
    over = _selection(wl, 5, k)
    over[0, :k] = first[0, :k]                       # query 0's rows are all resident (hits)
    hc.fetch(sa.batch, over.cuda(), k, slots)
    assert lib.check_device_error() == lib.DSA_ERR_CAPACITY
    assert hc.resident() == before
    st = hc.stats()
    assert st["overflow"] == 1 and st["misses"] == 0 and st["steps"] == 2
    s = slots.cpu()
    rows = _entry_rows(wl_cpu, over)
    assert (s[0][rows[0] >= 0] >= 0).all()           # hits still resolve
    assert (s[1:] == -1).all()                       # misses do not
    # a fitting step afterwards proceeds as if the failed one never happened
    lru = oracle.HiSparseLRU(5000)
    lru.step(_oracle_rows(wl_cpu, first))
    nxt = _selection(wl, 7, k)
    nxt[2:] = -1
    hc.fetch(sa.batch, nxt.cuda(), k, slots)
    assert lib.check_device_error() == lib.DSA_OK
    hits, misses, evicted = lru.step(_oracle_rows(wl_cpu, nxt))
    assert hc.resident() == list(lru.order)
    assert hc.stats()["misses"] == len(misses) and hc.stats()["evicted"] == len(evicted)


def test_unpinned_host_pool_is_rejected(lib):
    spec = W.SPECS["decode"].scaled(batch=2, ctx_len=3000)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    pageable = wl.kv[0].cpu()
    cap = 4096
    pool = torch.empty((cap, spec.d_qk), dtype=torch.bfloat16, device="cuda")
    state = torch.empty(lib.hisparse_state_bytes(cap, pageable.shape[0]), dtype=torch.uint8, device="cuda")
    hs = lib.make_hisparse(pool, pageable.shape[0], state)
    lib.hisparse_reset(hs)
    host_cache = lib.make_cache(pageable, wl.seq_start)
    slots = torch.empty((wl.total_q, spec.topk), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.DsaError) as e:
        lib.hisparse_fetch(hs, sa.batch, host_cache, sa.idx, spec.topk, slots, sa.workspace)
    assert e.value.status == lib.DSA_ERR_INVALID_ARG


def test_full_size_decode_trace(lib):
    # the decode workload (32 x 32768, top-2048): layer 0's 1,048,576 rows in pinned
    # host memory, 262,144 HBM slots; the indexer's selection, then decode-like
    # steps that replace every eighth entry
    spec = W.SPECS["decode"]
    capacity = 262144
    wl, sa, host, hc = _setup(lib, spec, capacity)
    wl_cpu = wl.to("cpu", kv_too=False)
    k, T = spec.topk, wl.total_q
    idx0, _, _ = sa.forward()
    sel = idx0.clone()
    g = torch.Generator(device="cuda").manual_seed(5)
    n = wl.seq_lens.to(torch.int64).view(T, 1)
    slots = torch.empty((T, k), dtype=torch.int32, device="cuda")
    lru = oracle.HiSparseLRU(capacity)
    out_a = torch.empty_like(sa.outs[0])
    out_b = torch.empty_like(sa.outs[0])
    for step in range(1, 5):
        if step > 1:
            fresh = (torch.rand((T, k), generator=g, device="cuda") * n).to(torch.int32)
            sel[:, ::8] = fresh[:, ::8]
        hc.fetch(sa.batch, sel, k, slots)
        assert lib.check_device_error() == lib.DSA_OK
        hits, misses, evicted = lru.step(_oracle_rows(wl_cpu, sel.cpu()))
        assert hc.stats() == dict(steps=step, requested=len(hits) + len(misses), hits=len(hits),
                                  misses=len(misses), evicted=len(evicted), overflow=0), f"step {step}"
        assert hc.resident() == list(lru.order), f"step {step}: LRU order"
        lib.sparse_mla_fwd(sa.batch, sa.layers[0], sel, k, out_a, None, sa.workspace)
        lib.sparse_mla_fwd(sa.batch, hc.layer(wl.q[0], spec.d_v, spec.scale), slots, k, out_b, None, sa.workspace)
        torch.cuda.synchronize()
        assert lib.check_device_error() == lib.DSA_OK
        assert torch.equal(out_a, out_b), f"step {step}"
