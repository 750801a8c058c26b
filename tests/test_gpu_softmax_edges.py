"""Sparse MLA when the logits rise or fall by large steps along the selection.

The kernel takes probabilities against a per-head reference that moves only
when a score passes it by more than 2^16; the first tile of a block always
moves it, a later tile moves it only when its logits jump.  Ordinary inputs
(N(0,1)*0.05 queries and latents) never make a later tile jump, so these cases
build the jump into the rope dims of the latent rows, which enter Q.K but not
the value (values are the first 512 dims), so outputs keep ordinary
magnitudes:

  C[s, 512] = step * (tile of s along the index row)   (a staircase)
  C[s, 513] = small integer per row                      (within-tile spread)
  Q[t, h, 512] = Q[t, h, 513] = 16 for the heads that see the staircase, else 0

With scale 1/16 a head that sees the staircase has logits step * tile + spread
(natural log units); a step of 12 is 17.3 in log2 units, past the 2^16 rule.

Every head is checked on its own against the float64 oracle over the same
index set (max |err| <= 1e-2 * max |ref| and mean |err| <= 1e-3 * max |ref|,
per head, stricter than per query), and LSE to 1e-4.
"""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from helpers import OUT_MAX_REL, OUT_MEAN_REL, make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


def _per_head_check(got, ref, what):
    for h in range(ref.shape[0]):
        err = np.abs(got[h].astype(np.float64) - ref[h])
        m = np.abs(ref[h]).max()
        assert err.max() <= OUT_MAX_REL * m, f"{what} head {h}: max err {err.max():.3e} vs {m:.3e}"
        assert err.mean() <= OUT_MEAN_REL * m, f"{what} head {h}: mean err {err.mean():.3e} vs {m:.3e}"


def _run_staircase(lib, step, heads_up, ctx=9000, batch=2, n_sel=2048, seed=61, holes=False):
    spec = W.SPECS["decode"].scaled(batch=batch, ctx_len=ctx, seed=seed)
    wl = W.make_workload(spec, device="cuda")
    T, k = wl.total_q, spec.topk
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for t in range(T):
        sel = torch.sort(torch.randperm(ctx, generator=g)[:n_sel]).values
        rows = W.pool_rows(wl, t, sel)
        tile = torch.arange(n_sel) // 128
        spread = torch.randint(0, 4, (n_sel,), generator=g).float()
        kv = wl.kv[0]
        kv[rows.cuda(), 512] = (step * tile.float()).to(torch.bfloat16).cuda()
        kv[rows.cuda(), 513] = spread.to(torch.bfloat16).cuda()
        if holes:
            sel = sel.clone()
            sel[5::31] = -1
        idx[t, :n_sel] = sel.to(torch.int32)
        q = wl.q[0]
        q[t, :, 512] = 0
        q[t, :, 513] = 0
        for h in heads_up:
            q[t, h, 512] = 16.0
            q[t, h, 513] = 16.0
    idx = idx.cuda()
    sa = make_sa(wl)
    out = torch.empty((T, spec.heads, spec.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, spec.heads), dtype=torch.float32, device="cuda")
    lib.sparse_mla_fwd(sa.batch, sa.layers[0], idx, k, out, lse, sa.workspace)
    assert lib.check_device_error() == lib.DSA_OK
    cpu = wl.to("cpu")
    for t in range(T):
        o, l = oracle.attention_on_set(cpu, t, 0, idx[t].cpu().numpy())
        _per_head_check(out[t].float().cpu().numpy(), o, f"step {step} query {t}")
        np.testing.assert_allclose(lse[t].cpu().numpy(), l, rtol=1e-4, atol=1e-4, err_msg=f"step {step} lse")
        if step > 0 and heads_up:
            # the staircase dominates: the head's LSE sits near the top step
            top = step * (n_sel // 128 - 1)
            assert l[heads_up[0]] > top, "the staircase did not reach the oracle"
    return out, lse


@pytest.mark.parametrize("heads_up", [[0], [37], list(range(64))], ids=["head0", "head37", "all"])
def test_rising_logits_move_the_reference_on_later_tiles(lib, heads_up):
    # 12 nats per 128-row tile: every later tile of every block passes the
    # reference by more than 2^16; the other heads stay flat, so the overflow
    # vote is raised by a few threads only and must leave them unscaled
    _run_staircase(lib, 12.0, heads_up)


def test_rising_logits_with_holes_and_a_partial_last_tile(lib):
    # -1 holes inside tiles and 1900 selected rows (a last tile of 108 rows)
    _run_staircase(lib, 12.0, [0, 1, 63], n_sel=1900, holes=True, seed=62)


def test_falling_logits_keep_the_first_reference(lib):
    # the first tile holds the maximum; later tiles never move the reference
    # and contribute with tiny weights
    _run_staircase(lib, -12.0, list(range(64)), seed=63)


def test_small_steps_below_the_rescale_threshold(lib):
    # 8 nats per tile (11.5 in log2 units): the reference stays put while the
    # probabilities grow up to 2^11.5 per tile, summed in fp32
    _run_staircase(lib, 8.0, [5, 40], seed=64)
