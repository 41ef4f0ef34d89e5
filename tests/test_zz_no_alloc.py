"""The backward's no-allocation entry point (dsv_sparse_attn_bwd_noalloc).

It exists for callers that cannot allocate device memory themselves: a framework that
owns all GPU memory through its own pool, a plug-in with a memory budget fixed at start,
or a latency-critical loop that must not call cudaMalloc/cudaFree.  It uses a fixed scratch
array inside the library instead of a caller workspace, so its results must match the
ordinary backward's, call after call, although every call reuses the same array.

This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import pytest
import torch

from dynamic_sparse_attention_estimate_gb300 import dsv_estimate_topk, dsv_sparse_attn_bwd, dsv_sparse_attn_fwd
from dynamic_sparse_attention_estimate_gb300.binding import dsv_last_device_status, load_library, make_dims
from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, Workload, make_inputs

from gpu_helpers import need_gpu


def _noalloc(lib, dims, g, o, lse, idx, out):
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dsv_sparse_attn_bwd_noalloc(ctypes.byref(dims), ptr(g["do"]), ptr(g["q"]), ptr(g["k"]), ptr(g["v"]),
                                           ptr(o), ptr(lse), ptr(idx), ptr(out[0]), ptr(out[1]), ptr(out[2]), stream)


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [WORKLOADS["tiny"], Workload("ragged", 1, 2, (5, 16, 16), 128, 32, 100, None, lr_max=8)],
                         ids=["tiny", "ragged-d128"])
def test_noalloc_backward_matches_the_workspace_backward_on_two_calls(wl):
    dev = need_gpu()
    g = {k: v.to(dev) for k, v in make_inputs(wl).items()}
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    ref = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
    torch.cuda.synchronize()
    lib = load_library()
    dims = make_dims(wl.B, wl.H, wl.N, wl.d, wl.r, wl.k)
    for call in range(2):
        out = tuple(torch.full_like(g["q"], float("nan")) for _ in range(3))
        status = _noalloc(lib, dims, g, o, lse, idx, out)
        assert status == 0, lib.dsv_last_error_message()
        torch.cuda.synchronize()
        assert dsv_last_device_status() == 0
        # the backward gives bitwise the same gradients whatever its wave plan, so the outputs
        # must be equal, not just close
        for name, got, want in zip(("dQ", "dK", "dV"), out, ref):
            assert torch.equal(got, want), f"{name} (call {call + 1}) differs from the workspace backward"

