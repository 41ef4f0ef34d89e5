"""The backward split in two calls (the rank structure of idx first, the rest after) gives bitwise
the same dQ, dK, dV as the one-call backward, also when the first part runs on a second stream
beside the forward."""
import pytest
import torch

from dynamic_sparse_attention_estimate_gb300 import (dsv_estimate_topk, dsv_sparse_attn_bwd,
                                                     dsv_sparse_attn_bwd_prepare, dsv_sparse_attn_bwd_prepared,
                                                     dsv_sparse_attn_fwd)
from dynamic_sparse_attention_estimate_gb300.binding import (dsv_last_device_status, dsv_sparse_attn_bwd_workspace,
                                                             make_dims)
from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,heads", [("tiny", 2), ("short", 2)])
def test_split_backward_is_bitwise_the_one_call_backward(name, heads):
    dev = need_gpu()
    wl = WORKLOADS[name].with_heads(heads)
    g = {n: t.to(dev) for n, t in make_inputs(wl).items()}
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    want = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)

    ws = torch.empty(dsv_sparse_attn_bwd_workspace(make_dims(wl.B, wl.H, wl.N, wl.d, wl.r, wl.k)),
                     dtype=torch.uint8, device=dev)
    ws.fill_(0xA5)                                   # stale bytes must not matter
    side = torch.cuda.Stream()
    have_idx, prepared = torch.cuda.Event(), torch.cuda.Event()
    idx2 = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    have_idx.record()
    o2, lse2 = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx2)     # enqueued before the prep
    with torch.cuda.stream(side):
        side.wait_event(have_idx)
        dsv_sparse_attn_bwd_prepare(idx2, wl.d, ws)
        prepared.record(side)
    torch.cuda.current_stream().wait_event(prepared)
    got = dsv_sparse_attn_bwd_prepared(g["do"], g["q"], g["k"], g["v"], o2, lse2, idx2, ws)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    assert torch.equal(idx, idx2) and torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b, n in zip(got, want, ("dQ", "dK", "dV")):
        assert torch.equal(a, b), n
