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
    lib.cache_append(sa.batch, new_k, sa.indexer.k, sa.workspace)
    for layer, c in zip(sa.layers, new_c):
        lib.cache_append(sa.batch, c, layer.kv, sa.workspace)
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
    lib.cache_append(sa.batch, rows, sa.indexer.k, sa.workspace)
    assert lib.check_device_error() == lib.DSA_ERR_BAD_INDEX
    changed = (wl.k_idx != before).any(dim=1).nonzero().flatten().cpu().tolist()
    assert len(changed) == wl.total_q - 1        # every other token was written
