"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Selection must be bit-exact; O, dQ, dK, dV (bf16) within max-abs 2e-2 and rel-L2 1e-2
of the oracle; LSE within 1e-2.  Small workloads are compared element by element;
the short-clip workload (the one the benchmark times) is compared on every head for
the selection, on whole heads for the forward, on sampled blocks for the backward
(dO zeroed outside them), and through closed-form invariants on every head.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_sparse_attention_estimate_gb300 import dsv_estimate_topk, dsv_sparse_attn_bwd, dsv_sparse_attn_fwd
from dynamic_sparse_attention_estimate_gb300.binding import dsv_last_device_status, dsv_sparse_attn_bwd_workspace, \
    make_dims
from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, Workload, make_inputs, sample_blocks

from gpu_helpers import EDGE_REL_ELEM, LSE_MAX_ABS, assert_close, check_idx_invariants, need_gpu, np64

pytestmark = pytest.mark.gpu


def _to(dev, x):
    return {k: v.to(dev) for k, v in x.items()}


def _run(g, k, workspace=None):
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    dq, dk, dv = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx, workspace=workspace)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    return idx, o, lse, dq, dk, dv


def _full_check(x, out, k, heads=None, rel_elem=0.0):
    idx, o, lse, dq, dk, dv = out
    B, H = x["q"].shape[:2]
    for h in (range(H) if heads is None else heads):
        c = {key: val[0, h] for key, val in x.items()}
        want = oracle.estimate_topk(c["q_lr"], c["k_lr"], 64, k)
        got = idx[0, h].cpu().numpy()
        assert np.array_equal(got, want), f"head {h}: selection differs in {(got != want).any(axis=1).sum()} blocks"
        ro, rl = oracle.sparse_attn_fwd(c["q"], c["k"], c["v"], want, 64)
        rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], want, 64, o=ro, lse=rl)
        assert_close(f"O[h{h}]", o[0, h], ro, rel_elem=rel_elem)
        assert_close(f"LSE[h{h}]", lse[0, h], rl, max_abs=LSE_MAX_ABS)
        assert_close(f"dQ[h{h}]", dq[0, h], rdq, rel_elem=rel_elem)
        assert_close(f"dK[h{h}]", dk[0, h], rdk, rel_elem=rel_elem)
        assert_close(f"dV[h{h}]", dv[0, h], rdv, rel_elem=rel_elem)


def test_tiny_workload_full():
    dev = need_gpu()
    wl = WORKLOADS["tiny"]
    x = make_inputs(wl)
    out = _run(_to(dev, x), wl.k)
    _full_check(x, out, wl.k)


def test_ragged_d128_r32_nb_not_multiple_of_16():
    """N = 1280 (20 blocks), d = 128, r = 32, k = 100 (a ragged last chunk), factors in [-8, 8]."""
    dev = need_gpu()
    wl = Workload("ragged", 1, 2, (5, 16, 16), 128, 32, 100, None, lr_max=8)
    x = make_inputs(wl)
    out = _run(_to(dev, x), wl.k)
    _full_check(x, out, wl.k)


@pytest.mark.parametrize("k", [1, 63, 65, 1024])
def test_edge_k_values(k):
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(1)
    x = make_inputs(wl)
    out = _run(_to(dev, x), k)
    _full_check(x, out, k, rel_elem=EDGE_REL_ELEM)
    if k == wl.N:
        assert torch.equal(out[0][0, 0].cpu(), torch.arange(wl.N, dtype=torch.int32).expand(wl.NB, wl.N))


def test_full_density_equals_dense_attention():
    """k = N: the sparse path is dense bidirectional attention (checked against SDPA too)."""
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(2)
    x = make_inputs(wl)
    g = _to(dev, x)
    idx, o, lse, dq, dk, dv = _run(g, wl.N)
    ref = torch.nn.functional.scaled_dot_product_attention(g["q"].float(), g["k"].float(), g["v"].float())
    assert_close("O vs SDPA", o, np64(ref))


@pytest.mark.parametrize("d", [64, 128])
def test_dense_path_with_a_partial_key_tile(d):
    """k = N runs the dense backward (key tiles of 128 accumulate dK and dV on chip; dQ per query
    block; no idx read, no partial rows).  N = 448 leaves the last key tile half full: the keys
    past N must get no probability and no gradient row."""
    dev = need_gpu()
    wl = Workload("dense448", 1, 2, (7, 8, 8), d, 16, 448, None)
    x = make_inputs(wl)
    out = _run(_to(dev, x), wl.N)
    _full_check(x, out, wl.N, rel_elem=EDGE_REL_ELEM)


def test_dense_backward_repeats_bitwise():
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(2)
    g = _to(dev, make_inputs(wl))
    a = _run(g, wl.N)
    b = _run(g, wl.N)
    for name, x, y in zip(("dQ", "dK", "dV"), a[3:], b[3:]):
        assert torch.equal(x, y), name


def test_ties_go_to_the_lower_key_index():
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(2)
    x = make_inputs(wl)
    x["k_lr"][0, 0].zero_()                      # every score 0: first k keys
    x["k_lr"][0, 1] = x["k_lr"][0, 1].clamp(-1, 1)  # few distinct scores: many ties
    out = _run(_to(dev, x), 200)
    assert torch.equal(out[0][0, 0].cpu(), torch.arange(200, dtype=torch.int32).expand(wl.NB, 200))
    _full_check(x, out, 200)


def test_selection_signed_zero_and_negative_thresholds():
    """Scores of a few distinct integer values with many ties, signed zeros among them (the
    selection compares scores against float bounds equivalent to their order keys, which fold -0
    into +0), and k cutting the ranking inside the zero group, in the negative values and near N:
    the selected sets equal the oracle's for every block."""
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(2)
    x = make_inputs(wl)
    gen = torch.Generator().manual_seed(5)
    vals = torch.tensor([-3.0, -2.0, -1.0, -0.0, 0.0, 1.0, 2.0, 3.0], dtype=torch.bfloat16)
    for h in range(2):
        x["k_lr"][0, h] = vals[torch.randint(0, 8, (wl.N, wl.r), generator=gen)]
        x["q_lr"][0, h] = torch.randint(-1, 2, (wl.N, wl.r), generator=gen).to(torch.bfloat16)
    x["q_lr"][0, 1, :64] = 0.0
    x["q_lr"][0, 1, 0, 0] = 1.0   # block 0 of head 1: s = K_lr[:, 0], signed zeros included
    g = _to(dev, x)
    for k in (1, 100, 500, 511, 512, 513, 700, 1000, 1023):
        idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], k)
        torch.cuda.synchronize()
        assert dsv_last_device_status() == 0
        for h in range(2):
            want = oracle.estimate_topk(x["q_lr"][0, h], x["k_lr"][0, h], 64, k)
            assert np.array_equal(idx[0, h].cpu().numpy(), want), f"k={k} head {h}"


def test_short_clip_selection_every_head_bit_exact():
    dev = need_gpu()
    wl = WORKLOADS["short"]
    x = make_inputs(wl)
    g = _to(dev, x)
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    torch.cuda.synchronize()
    check_idx_invariants(idx, wl.N)
    for h in range(wl.H):
        want = oracle.estimate_topk(x["q_lr"][0, h], x["k_lr"][0, h], 64, wl.k)
        assert np.array_equal(idx[0, h].cpu().numpy(), want), f"head {h}"


def test_short_clip_selection_r32_two_row_tiles():
    """12 heads x 256 query blocks with r = 32: the estimate runs 22 query blocks per CTA on two m16
    row tiles (one wave over the SMs); every head's selection equals the oracle's."""
    import dataclasses
    dev = need_gpu()
    wl = dataclasses.replace(WORKLOADS["short"], r=32)
    x = make_inputs(wl)
    g = _to(dev, x)
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    torch.cuda.synchronize()
    check_idx_invariants(idx, wl.N)
    for h in range(wl.H):
        want = oracle.estimate_topk(x["q_lr"][0, h], x["k_lr"][0, h], 64, wl.k)
        assert np.array_equal(idx[0, h].cpu().numpy(), want), f"head {h}"


def test_short_clip_attention():
    dev = need_gpu()
    wl = WORKLOADS["short"]
    x = make_inputs(wl)
    g = _to(dev, x)
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    dq, dk, dv = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    idx_np = idx.cpu().numpy()
    # forward on two whole heads
    for h in (0, wl.H - 1):
        ro, rl = oracle.sparse_attn_fwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], idx_np[0, h], 64)
        assert_close(f"O[h{h}]", o[0, h], ro)
        assert_close(f"LSE[h{h}]", lse[0, h], rl, max_abs=LSE_MAX_ABS)
    # closed forms on every head of the unmasked backward
    for h in range(wl.H):
        sdo = np64(g["do"][0, h]).sum(0)
        assert_close(f"sum dV[h{h}] = sum dO", np64(dv[0, h]).sum(0), sdo, max_abs=0.5, rel_l2=1e-2)
        sel = np.zeros(wl.N, bool)
        sel[np.unique(idx_np[0, h])] = True
        assert not np64(dk[0, h])[~sel].any() and not np64(dv[0, h])[~sel].any()
        assert np.abs(np64(dk[0, h]).sum(0)).max() < 0.5
    # backward on sampled blocks: dO zeroed outside them, every head
    blocks = sample_blocks(wl.NB, 16)
    mask = torch.zeros(wl.N, dtype=torch.bool)
    for b in blocks:
        mask[b * 64:(b + 1) * 64] = True
    do_m = g["do"] * mask.to(dev)[None, None, :, None]
    dq2, dk2, dv2 = dsv_sparse_attn_bwd(do_m, g["q"], g["k"], g["v"], o, lse, idx)
    torch.cuda.synchronize()
    rows = mask.numpy()
    for h in range(wl.H):
        c = {key: val[0, h] for key, val in x.items()}
        rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], idx_np[0, h], 64, blocks=blocks)
        assert_close(f"dQ[h{h}] sampled", np64(dq2[0, h])[rows], rdq[rows])
        assert_close(f"dK[h{h}] sampled", dk2[0, h], rdk)
        assert_close(f"dV[h{h}] sampled", dv2[0, h], rdv)


def test_backward_is_deterministic_and_wave_independent():
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(2)
    x = make_inputs(wl)
    g = _to(dev, x)
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    ref = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
    again = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
    dims = make_dims(1, 2, wl.N, wl.d, wl.r, wl.k)
    small = dsv_sparse_attn_bwd_workspace(dims, minimum=True)
    for nbytes in (small, small * 2, small * 3, small * 5, small * 12, small * 40):  # sub-head waves of a few blocks
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        other = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx, workspace=ws)
        for a, b in zip(ref, other):
            assert torch.equal(a, b)
    for a, b in zip(ref, again):
        assert torch.equal(a, b)
    assert dsv_last_device_status() == 0


def test_backward_with_unordered_idx_rows_matches_ascending():
    """The backward does not need ascending idx rows (only distinct keys): its bitmap kernel walks
    ascending rows once and falls back to filtering every row per key tile when a row is out of
    order.  Rows reversed or rotated give the same dK and dV bit for bit (each (block, key)
    contribution is the same product and every key's contributions are summed in block order) and
    dQ up to the order of its fp32 accumulation over chunks; also across sub-head waves."""
    dev = need_gpu()
    for wl in (WORKLOADS["tiny"].with_heads(2), Workload("ragged", 1, 2, (5, 16, 16), 128, 32, 100, None, lr_max=8)):
        g = _to(dev, make_inputs(wl))
        idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
        o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
        ref = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
        small = dsv_sparse_attn_bwd_workspace(make_dims(1, wl.H, wl.N, wl.d, wl.r, wl.k), minimum=True)
        for perm in (idx.flip(-1).contiguous(), torch.roll(idx, 37, dims=-1).contiguous()):
            for ws in (None, torch.empty(small * 3, dtype=torch.uint8, device=dev)):
                dq, dk, dv = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, perm, workspace=ws)
                assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
                err = (dq.float() - ref[0].float()).abs().max().item()
                assert err <= 1e-2 * ref[0].float().abs().max().item() + 1e-3, err
        assert dsv_last_device_status() == 0


def test_backward_tile_bounds_path_matches_the_general_path():
    """Over many key tiles (here nine, the last one partial) the backward's bitmap kernel reads only
    each ascending row's run per tile, from tile bounds found by a first pass; rows out of order take
    the general method.  The same rows ascending and reversed must give the same dK and dV bit for
    bit, in one wave and across sub-head waves (whose bounds start at a block offset)."""
    dev = need_gpu()
    wl = Workload("tiles", 1, 1, (17, 128, 128), 64, 16, 96, (4, 4, 4))
    assert (wl.N + 32767) // 32768 == 9
    g = _to(dev, make_inputs(wl))
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    small = dsv_sparse_attn_bwd_workspace(make_dims(1, 1, wl.N, wl.d, wl.r, wl.k), minimum=True)
    for ws in (None, torch.empty(small + 30_000_000, dtype=torch.uint8, device=dev)):  # waves of ~1,000 blocks
        asc = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx, workspace=ws)
        rev = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx.flip(-1).contiguous(), workspace=ws)
        assert torch.equal(asc[1], rev[1]) and torch.equal(asc[2], rev[2])
        err = (asc[0].float() - rev[0].float()).abs().max().item()
        assert err <= 1e-2 * asc[0].float().abs().max().item() + 1e-3, err
    assert dsv_last_device_status() == 0


def test_out_of_range_and_repeated_indices_set_the_device_status():
    dev = need_gpu()
    wl = WORKLOADS["tiny"].with_heads(1)
    g = _to(dev, make_inputs(wl))
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    bad = idx.clone()
    bad[0, 0, 3, 5] = wl.N + 7          # out of range: skipped, flagged
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], bad)
    assert dsv_last_device_status() == 5
    assert dsv_last_device_status() == 0  # read clears it
    dup = idx.clone()
    dup[0, 0, 2, 1] = dup[0, 0, 2, 0]    # repeated key in one row
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, dup)
    assert dsv_last_device_status() == 5


def test_multi_wave_backward_matches_one_wave_bitwise():
    """The short clip's backward through workspaces that hold a whole head, part of a head, or a
    few blocks per wave (waves whose rank structure is built on a second stream while the previous
    wave is reduced, where the workspace has room for two copies of it): bitwise the one-wave
    gradients."""
    dev = need_gpu()
    wl = WORKLOADS["short"].with_heads(3)
    g = _to(dev, make_inputs(wl))
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    ref = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx)
    dims = make_dims(1, 3, wl.N, wl.d, wl.r, wl.k)
    rec = dsv_sparse_attn_bwd_workspace(dims)
    for frac in (0.6, 0.34, 0.2, 0.07, 0.03):
        ws = torch.empty(int(rec * frac) // 256 * 256, dtype=torch.uint8, device=dev)
        other = dsv_sparse_attn_bwd(g["do"], g["q"], g["k"], g["v"], o, lse, idx, workspace=ws)
        for a, b in zip(ref, other):
            assert torch.equal(a, b), f"workspace fraction {frac}"
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
