"""Python front end on the GPU: result buffers supplied by the caller (views
of one staging buffer, as a server lays them out) and the overlapped forward
without events give dsa_forward's results bit for bit."""
import pytest
import torch

import dsa_workloads as W
from helpers import make_sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from long_context_lightning_gb300 import _lib
    return _lib


@pytest.mark.parametrize("name,kw", [("decode", dict(batch=6, ctx_len=7000)),
                                     ("indexshare", dict(batch=2, ctx_len=9000))])
def test_results_into_caller_buffers(lib, name, kw):
    from long_context_lightning_gb300 import SparseAttention
    spec = W.SPECS[name].scaled(**kw)
    wl = W.make_workload(spec, device="cuda")
    ref = make_sa(wl)
    idx_ref, outs_ref, lses_ref = ref.forward()
    T, L, H = wl.total_q, spec.n_layers, spec.heads
    # one byte buffer: idx, then each layer's output, then each layer's LSE (256-byte aligned pieces)
    sizes = [T * spec.topk * 4] + [T * H * spec.d_v * 2] * L + [T * H * 4] * L
    offs, n = [], 0
    for sz in sizes:
        offs.append(n)
        n += (sz + 255) // 256 * 256
    arena = torch.full((n,), 0x7F, dtype=torch.uint8, device="cuda")
    view = lambda i, dt, shape: arena[offs[i]:offs[i] + sizes[i]].view(dt).view(shape)  # noqa: E731
    idx = view(0, torch.int32, (T, spec.topk))
    outs = [view(1 + l, torch.bfloat16, (T, H, spec.d_v)) for l in range(L)]
    lses = [view(1 + L + l, torch.float32, (T, H)) for l in range(L)]
    sa = SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, spec.d_v,
                         spec.scale, spec.topk, seq_start=wl.seq_start, idx=idx, outs=outs, lses=lses)
    got_idx, got_outs, got_lses = sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    assert got_idx.data_ptr() == idx.data_ptr()
    assert torch.equal(idx, idx_ref)
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a, b)
    for a, b in zip(lses, lses_ref):
        assert torch.equal(a, b)
    # the overlapped entry point with no events is the plain forward
    for x in (idx, *outs, *lses):
        x.zero_()
    sa.forward_overlapped()
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref)
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a, b)


def test_outputs_into_pinned_host_memory(lib):
    # the sparse MLA writes outputs and LSE straight into pinned host memory
    # (no copy back); they equal the device-memory results bit for bit
    from long_context_lightning_gb300 import SparseAttention
    spec = W.SPECS["ragged"].scaled(batch=7, ctx_range=(300, 6000))
    wl = W.make_workload(spec, device="cuda")
    ref = make_sa(wl)
    idx_ref, outs_ref, lses_ref = ref.forward()
    outs = [torch.full(o.shape, -1.0, dtype=o.dtype).pin_memory() for o in outs_ref]
    lses = [torch.full(x.shape, -1.0, dtype=x.dtype).pin_memory() for x in lses_ref]
    sa = SparseAttention(wl.cu_seqlens_q, wl.seq_lens, wl.q_idx, wl.w, wl.k_idx, wl.q, wl.kv, spec.d_v, spec.scale,
                         spec.topk, page_table=wl.page_table, page_size=spec.page_size, outs=outs, lses=lses)
    sa.forward()
    torch.cuda.synchronize()
    assert lib.check_device_error() == lib.DSA_OK
    assert torch.equal(sa.idx, idx_ref)
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a, b.cpu())
    for a, b in zip(lses, lses_ref):
        assert torch.equal(a, b.cpu())
