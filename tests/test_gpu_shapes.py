"""Shapes away from the benchmark configs, on the GPU against the float64
oracle: attention heads 1..64 at the 576-dim latent (MMA N padded past the
heads), indexer heads between the two tile widths (16 and 64) and head dims
32 / 64 / 128, top-k sizes that leave a partial 128-row tile, and query
groups with a partial tail (five queries per sequence: groups of four)."""
import pytest

import dsa_workloads as W
from helpers import compare_forward, make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


@pytest.mark.parametrize("heads,idx_heads,idx_dim,topk,q_per_seq,ctx", [
    (1, 1, 32, 100, 1, 2600),
    (20, 24, 64, 777, 1, 4100),
    (33, 50, 128, 2000, 3, 5000),
    (64, 7, 128, 1500, 5, 3900),
])
def test_off_config_shapes_match_oracle(lib, heads, idx_heads, idx_dim, topk, q_per_seq, ctx):
    spec = W.SPECS["decode"].scaled(batch=3, ctx_len=ctx, heads=heads, idx_heads=idx_heads, idx_dim=idx_dim,
                                    topk=topk, q_per_seq=q_per_seq)
    wl = W.make_workload(spec, device="cuda")
    idx, outs, lses = make_sa(wl).forward()
    assert lib.check_device_error() == lib.DSA_OK
    compare_forward(wl.to("cpu"), idx, outs, lses, range(wl.total_q))
