"""The sparse-MLA entry point for callers that cannot pass a workspace.

Such callers (a plugin interface that only hands over tensor pointers, or an
engine whose device memory is all taken by its own pool) get the per-call plan
from a static device array inside the library.  This file is collected last so
that a run stopping at the first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import dsa_workloads as W
from helpers import OUT_MAX_REL, OUT_MEAN_REL, make_sa

pytestmark = pytest.mark.gpu


def _close(got, ref, what):
    got = got.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    m = np.abs(ref).max()
    assert err.max() <= OUT_MAX_REL * m, f"{what}: max err {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_REL * m, f"{what}: mean err {err.mean():.3e}"


def test_noalloc_matches_workspace_entry_point_twice():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib

    # two different problems in a row, so the second call must not depend on
    # what the first one left in the shared static array
    for call, (batch, ctx) in enumerate([(6, 5000), (3, 9000)]):
        spec = W.SPECS["decode"].scaled(batch=batch, ctx_len=ctx, seed=50 + call)
        wl = W.make_workload(spec, device="cuda")
        sa = make_sa(wl)
        idx, outs, lses = sa.forward()              # an index set from the fused path
        ref = torch.empty_like(outs[0])
        ref_lse = torch.empty_like(lses[0])
        _lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx, spec.topk, ref, ref_lse, sa.workspace)
        got = torch.full_like(outs[0], 3.0)
        got_lse = torch.full_like(lses[0], 3.0)
        _lib.sparse_mla_fwd_noalloc(sa.batch, sa.layers[0], idx, spec.topk, got, got_lse)
        assert _lib.check_device_error() == _lib.DSA_OK
        _close(got, ref, f"call {call}: output")
        np.testing.assert_allclose(got_lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-4, atol=1e-4)


def test_noalloc_rejects_batches_beyond_its_static_scratch():
    from long_context_lightning_gb300 import _lib
    T = _lib.NOALLOC_MAX_QUERIES + 1
    cu = torch.arange(T + 1, dtype=torch.int32, device="cuda")
    lens = torch.full((T,), 4000, dtype=torch.int32, device="cuda")
    batch = _lib.make_batch(cu, lens, T, 4000, 1)
    spec = W.SPECS["decode"].scaled(batch=1, ctx_len=4000)
    wl = W.make_workload(spec, device="cuda")
    layer = make_sa(wl).layers[0]
    idx = torch.zeros((T, spec.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((T, spec.heads, spec.d_v), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.DsaError) as e:
        _lib.sparse_mla_fwd_noalloc(batch, layer, idx, spec.topk, out, None)
    assert e.value.status == _lib.DSA_ERR_UNSUPPORTED
