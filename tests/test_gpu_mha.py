"""MHA mode on the GPU against the float64 oracle: the per-head up-projection
of the latent rows (rope dims bit for bit), and attention of every head over
the GPU's own top-k selection, checked by the output rule; paged and ragged
batches, dense rows (context <= k) and sparse rows, empty selections and bad
indices."""
import numpy as np
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


def _mha(wl, layer=0):
    from long_context_lightning_gb300 import SparseMHA
    s = wl.spec
    m = SparseMHA(wl.cu_seqlens_q, wl.seq_lens, wl.kv[layer], wl.w_uk[layer], wl.w_uv[layer], s.scale,
                  seq_start=wl.seq_start, page_table=wl.page_table, page_size=s.page_size)
    m.project()
    return m


def test_projection_matches_oracle(lib):
    spec = W.SPECS["mha"].scaled(ctx_len=700, q_per_seq=10, heads=6)
    wl = W.make_workload(spec, device="cuda")
    m = _mha(wl)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    rows = torch.tensor([0, 1, 127, 128, 129, 350, 698, 699])
    c = oracle.bf16_to_f64(wl.kv[0][rows.cuda()])
    K, V = oracle.mha_upproject(c, oracle.bf16_to_f64(wl.w_uk[0]), oracle.bf16_to_f64(wl.w_uv[0]))
    H = spec.heads
    k_got = m.k_pool[rows.cuda()].view(len(rows), H, 256)
    v_got = m.v_pool[rows.cuda()].view(len(rows), H, 256)
    check_output(oracle.bf16_to_f64(k_got[:, :, :192]).reshape(-1, 192), K[:, :, :192].reshape(-1, 192), "keys")
    check_output(oracle.bf16_to_f64(v_got).reshape(-1, 256), V.reshape(-1, 256), "values")
    # the rope dims are the latent's own, copied to every head
    for h in range(H):
        assert torch.equal(k_got[:, h, 192:], wl.kv[0][rows.cuda()][:, 512:576])


@pytest.mark.parametrize("name,kw,queries", [
    ("small", dict(ctx_len=2500, q_per_seq=600, heads=4), None),
    ("paged_ragged", dict(batch=3, ctx_len=None, ctx_range=(1500, 5000), q_per_seq=150, heads=8, paged=True),
     None),
])
def test_attention_matches_oracle(lib, name, kw, queries):
    spec = W.SPECS["mha"].scaled(**kw)
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx, _, _ = sa.forward()
    m = _mha(wl)
    T = wl.total_q
    out = torch.empty((T, spec.heads, 256), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, spec.heads), dtype=torch.float32, device="cuda")
    m.forward(wl.q_mha[0], idx, spec.topk, out, lse)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    seq, pos = wl.query_positions()
    rng = np.random.default_rng(11)
    sample = sorted(set([0, T - 1] + rng.choice(T, size=min(T, 14), replace=False).tolist()))
    dense = sparse = 0
    cpu = wl.to("cpu")
    idx_c, out_c, lse_c = idx.cpu(), out.cpu(), lse.cpu()
    for t in sample:
        n = pos[t] + 1
        sel = idx_c[t, :min(n, spec.topk)].numpy()
        dense += n <= spec.topk
        sparse += n > spec.topk
        o, l = oracle.mha_attention_on_set(cpu, t, 0, sel)
        check_output(oracle.bf16_to_f64(out_c[t]), o, f"{name} query {t}")
        check_lse(lse_c[t].numpy(), l, f"{name} query {t}")
    assert sparse > 0
    if name == "small":
        assert dense > 0


def test_full_size_sample(lib):
    spec = W.SPECS["mha"]
    wl = W.make_workload(spec, device="cuda")
    sa = make_sa(wl)
    idx, _, _ = sa.forward()
    m = _mha(wl)
    T = wl.total_q
    out = torch.empty((T, spec.heads, 256), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, spec.heads), dtype=torch.float32, device="cuda")
    m.forward(wl.q_mha[0], idx, spec.topk, out, lse)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    seq, pos = wl.query_positions()
    cpu = wl.to("cpu")
    idx_c, out_c, lse_c = idx.cpu(), out.cpu(), lse.cpu()
    for t in (0, 511, 512, 1700, T - 1):      # dense (n <= 2048) and sparse rows
        sel = idx_c[t, :min(pos[t] + 1, spec.topk)].numpy()
        o, l = oracle.mha_attention_on_set(cpu, t, 0, sel)
        check_output(oracle.bf16_to_f64(out_c[t]), o, f"query {t}")
        check_lse(lse_c[t].numpy(), l, f"query {t}")


def test_empty_and_bad_selections(lib):
    spec = W.SPECS["mha"].scaled(ctx_len=600, q_per_seq=20, heads=2, topk=64)
    wl = W.make_workload(spec, device="cuda")
    m = _mha(wl)
    T = wl.total_q
    idx = torch.full((T, spec.topk), -1, dtype=torch.int32, device="cuda")
    idx[3, :5] = torch.tensor([0, 10, 20, 30, 40], dtype=torch.int32)
    out = torch.empty((T, spec.heads, 256), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, spec.heads), dtype=torch.float32, device="cuda")
    m.forward(wl.q_mha[0], idx, spec.topk, out, lse)
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    assert (out[0] == 0).all() and torch.isneginf(lse[0]).all()
    o, l = oracle.mha_attention_on_set(wl.to("cpu"), 3, 0, np.array([0, 10, 20, 30, 40]))
    check_output(oracle.bf16_to_f64(out[3].cpu()), o, "five rows")
    idx[5, 0] = 10 ** 6                            # beyond the context: flagged, skipped
    m.forward(wl.q_mha[0], idx, spec.topk, out, lse)
    assert lib.check_device_error() == lib.DSA_ERR_BAD_INDEX
    assert (out[5] == 0).all()
