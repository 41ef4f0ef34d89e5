"""GPU parity of the mass-based adaptive selection (through the C ABI) against the oracle.

Per query block k must equal the oracle's exactly (the decision is taken in integer weights
from the same fp32 recipe on both sides), and the CSR key lists must equal the oracle's
top-k of each block bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_sparse_attention_estimate_gb300 import dsv_estimate_mass_k, dsv_estimate_topk_csr
from dynamic_sparse_attention_estimate_gb300.binding import dsv_last_device_status, mass_parameters
from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, Workload, make_inputs

from gpu_helpers import need_gpu, np64

pytestmark = pytest.mark.gpu


def _select(g, tau, mass, with_order=False, dense_above=None):
    k_row, rowptr, order = dsv_estimate_mass_k(g["q_lr"], g["k_lr"], tau, mass, dense_above=dense_above)
    cols = dsv_estimate_topk_csr(g["q_lr"], g["k_lr"], k_row, rowptr)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    # the launch order: a permutation of the rows, by non-increasing number of 128-key chunks
    o = order.cpu().numpy()
    assert np.array_equal(np.sort(o), np.arange(o.size))
    nch = (k_row.cpu().numpy().reshape(-1)[o] + 127) // 128
    assert np.all(np.diff(nch) <= 0)
    out = (k_row.cpu().numpy(), rowptr.cpu().numpy(), cols.cpu().numpy())
    return out + (order,) if with_order else out


def _check_head(x, b, h, k_row, rowptr, cols, tau, mass, dense_num=0):
    tau_log2, mass_num = mass_parameters(tau, mass)
    s = oracle.block_scores(oracle.block_representatives(np64(x["q_lr"][b, h]), 64), np64(x["k_lr"][b, h]))
    want_k = oracle.mass_k(s, tau_log2, mass_num, dense_num)
    H, NB = k_row.shape[1], k_row.shape[2]
    assert np.array_equal(k_row[b, h], want_k), np.flatnonzero(k_row[b, h] != want_k)[:8]
    for blk in range(NB):
        row = (b * H + h) * NB + blk
        got = cols[rowptr[row]:rowptr[row + 1]]
        assert np.array_equal(got, oracle.topk_select(s[blk:blk + 1], int(want_k[blk]))[0]), (h, blk)


@pytest.mark.parametrize("tau,mass", [(1 / 64, 0.9), (0.05, 0.5), (0.01, 0.99), (1.0, 0.9), (0.002, 1.0)])
def test_mass_selection_tiny(tau, mass):
    need_gpu()
    wl = WORKLOADS["tiny"]
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols = _select(g, tau, mass)
    assert rowptr[0] == 0 and np.array_equal(np.diff(rowptr), k_row.reshape(-1))
    for h in range(wl.H):
        _check_head(x, 0, h, k_row, rowptr, cols, tau, mass)


def test_sparse_dense_switch_tiny():
    # blocks whose adaptive k exceeds 72 % of the keys take all of them (ascending)
    need_gpu()
    wl = WORKLOADS["tiny"]
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols = _select(g, 0.003, 0.9, dense_above=0.72)
    dense_num = int(round(0.72 * 65536))
    assert (k_row == wl.N).any() and (k_row < wl.N).any()    # both kinds of block occur
    for h in range(wl.H):
        _check_head(x, 0, h, k_row, rowptr, cols, 0.003, 0.9, dense_num)


def test_mass_selection_ragged_r32():
    need_gpu()
    wl = Workload("ragged_mass", 1, 2, (5, 16, 16), 128, 32, 100, None)   # N = 1280: 20 blocks
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols = _select(g, 0.02, 0.9)
    for h in range(wl.H):
        _check_head(x, 0, h, k_row, rowptr, cols, 0.02, 0.9)


def test_mass_selection_short_clip_two_heads():
    need_gpu()
    wl = WORKLOADS["short"].with_heads(2)
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols = _select(g, 1 / 64, 0.9)
    for h in range(wl.H):
        _check_head(x, 0, h, k_row, rowptr, cols, 1 / 64, 0.9)


def test_mass_selection_short_clip_every_head():
    """All 12 heads at once: the CSR top-k runs 22 query blocks per CTA on two m16 row tiles."""
    need_gpu()
    wl = WORKLOADS["short"]
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols = _select(g, 1 / 64, 0.9)
    for h in range(wl.H):
        _check_head(x, 0, h, k_row, rowptr, cols, 1 / 64, 0.9)


def _abs_contributions(c, lists, blocks):
    """Per key, the sum over blocks of |that block's contribution| to dK and dV: each block's
    contribution is one bf16 partial row, rounded once, so the rounding scales with these."""
    ak = np.zeros(tuple(c["k"].shape))
    av = np.zeros_like(ak)
    for b in blocks:
        _, dk_b, dv_b = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], lists, 64, blocks=[b])
        ak += np.abs(dk_b)
        av += np.abs(dv_b)
    return ak, av


def _assert_grad(name, got, ref, magnitude):
    from gpu_helpers import EDGE_REL_ELEM, MAX_ABS, REL_L2
    g = np64(got)
    err = np.abs(g - ref)
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    excess = float((err - (MAX_ABS + EDGE_REL_ELEM * magnitude)).max())
    assert excess <= 0 and rel <= REL_L2, f"{name}: max-abs {err.max():.3e}, excess {excess:.3e}, rel-L2 {rel:.3e}"


def _csr_lists(rowptr, cols, b, h, H, NB):
    return [cols[rowptr[(b * H + h) * NB + i]:rowptr[(b * H + h) * NB + i + 1]] for i in range(NB)]


def test_csr_attention_tiny_and_ragged():
    from dynamic_sparse_attention_estimate_gb300 import dsv_sparse_attn_bwd_csr, dsv_sparse_attn_fwd_csr
    from gpu_helpers import EDGE_REL_ELEM, LSE_MAX_ABS, assert_close
    need_gpu()
    # adaptive k gives some blocks very few keys, so gradients reach magnitudes where one bf16
    # spacing exceeds the absolute bound: the edge cases' magnitude-aware element bound, taken
    # on the sum of the blocks' |contributions| (each is one bf16 partial row)
    for wl, tau, mass in ((WORKLOADS["tiny"], 0.05, 0.9),
                          (Workload("ragged_mass", 1, 2, (5, 16, 16), 128, 32, 100, None), 0.02, 0.8)):
        x = make_inputs(wl)
        g = {k: v.cuda() for k, v in x.items()}
        k_row, rowptr, cols, order = _select(g, tau, mass, with_order=True)
        rp, cl = torch.from_numpy(rowptr).cuda(), torch.from_numpy(cols).cuda()
        o, lse = dsv_sparse_attn_fwd_csr(g["q"], g["k"], g["v"], rp, cl)
        dq, dk, dv = dsv_sparse_attn_bwd_csr(g["do"], g["q"], g["k"], g["v"], o, lse, rp, cl)
        # launch order changes nothing in the results
        o2, lse2 = dsv_sparse_attn_fwd_csr(g["q"], g["k"], g["v"], rp, cl, order=order)
        dq2, dk2, dv2 = dsv_sparse_attn_bwd_csr(g["do"], g["q"], g["k"], g["v"], o2, lse2, rp, cl, order=order)
        for a, b2 in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
            assert torch.equal(a, b2)
        torch.cuda.synchronize()
        assert dsv_last_device_status() == 0
        for h in range(wl.H):
            lists = _csr_lists(rowptr, cols, 0, h, wl.H, wl.NB)
            c = {key: val[0, h] for key, val in x.items()}
            ro, rl = oracle.sparse_attn_fwd(c["q"], c["k"], c["v"], lists, 64)
            assert_close(f"{wl.name} O[h{h}]", o[0, h], ro)
            assert_close(f"{wl.name} LSE[h{h}]", lse[0, h], rl, max_abs=LSE_MAX_ABS)
            rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], lists, 64)
            ak, av = _abs_contributions(c, lists, range(wl.NB))
            _assert_grad(f"{wl.name} dQ[h{h}]", dq[0, h], rdq, np.abs(rdq))
            _assert_grad(f"{wl.name} dK[h{h}]", dk[0, h], rdk, ak)
            _assert_grad(f"{wl.name} dV[h{h}]", dv[0, h], rdv, av)


def test_csr_attention_short_clip_two_heads():
    from dynamic_sparse_attention_estimate_gb300 import dsv_sparse_attn_bwd_csr, dsv_sparse_attn_fwd_csr
    from dynamic_sparse_attention_estimate_gb300.inputs import sample_blocks
    from gpu_helpers import EDGE_REL_ELEM, LSE_MAX_ABS, assert_close
    need_gpu()
    wl = WORKLOADS["short"].with_heads(2)
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    k_row, rowptr, cols, order = _select(g, 1 / 64, 0.9, with_order=True)
    rp, cl = torch.from_numpy(rowptr).cuda(), torch.from_numpy(cols).cuda()
    o, lse = dsv_sparse_attn_fwd_csr(g["q"], g["k"], g["v"], rp, cl, order=order)
    blocks = sample_blocks(wl.NB, 8)
    mask = torch.zeros(wl.N, dtype=torch.bool)
    for b in blocks:
        mask[b * 64:(b + 1) * 64] = True
    do_m = g["do"] * mask.cuda()[None, None, :, None]
    dq, dk, dv = dsv_sparse_attn_bwd_csr(do_m, g["q"], g["k"], g["v"], o, lse, rp, cl, order=order)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    rows = mask.numpy()
    for h in range(wl.H):
        lists = _csr_lists(rowptr, cols, 0, h, wl.H, wl.NB)
        c = {key: val[0, h] for key, val in x.items()}
        ro, rl = oracle.sparse_attn_fwd(c["q"], c["k"], c["v"], lists, 64, blocks=blocks)
        assert_close(f"O[h{h}] sampled", np64(o[0, h])[rows], ro[rows])
        assert_close(f"LSE[h{h}] sampled", np64(lse[0, h])[rows], rl[rows], max_abs=LSE_MAX_ABS)
        rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], lists, 64, blocks=blocks)
        ak, av = _abs_contributions(c, lists, blocks)
        _assert_grad(f"dQ[h{h}] sampled", dq[0, h][torch.from_numpy(rows)], rdq[rows], np.abs(rdq[rows]))
        _assert_grad(f"dK[h{h}] sampled", dk[0, h], rdk, ak)
        _assert_grad(f"dV[h{h}] sampled", dv[0, h], rdv, av)


def test_heterogeneous_per_head_k_in_one_launch():
    # a different k per head (100 and 700), all heads in one CSR launch, longest rows first
    from dynamic_sparse_attention_estimate_gb300 import dsv_sparse_attn_bwd_csr, dsv_sparse_attn_fwd_csr
    from dynamic_sparse_attention_estimate_gb300.binding import dsv_csr_launch_order
    from gpu_helpers import LSE_MAX_ABS, assert_close
    need_gpu()
    wl = WORKLOADS["tiny"]
    x = make_inputs(wl)
    g = {k: v.cuda() for k, v in x.items()}
    ks = (100, 700)
    k_row = torch.tensor([ks[h] for h in range(wl.H) for _ in range(wl.NB)], dtype=torch.int32).cuda()
    rowptr = torch.zeros(wl.H * wl.NB + 1, dtype=torch.int64)
    rowptr[1:] = torch.cumsum(k_row.cpu().to(torch.int64), 0)
    rowptr = rowptr.cuda()
    cols = dsv_estimate_topk_csr(g["q_lr"], g["k_lr"], k_row.view(1, wl.H, wl.NB), rowptr)
    order = dsv_csr_launch_order(rowptr, 1, wl.H, wl.N)
    o, lse = dsv_sparse_attn_fwd_csr(g["q"], g["k"], g["v"], rowptr, cols, order=order)
    dq, dk, dv = dsv_sparse_attn_bwd_csr(g["do"], g["q"], g["k"], g["v"], o, lse, rowptr, cols, order=order)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    od = order.cpu().numpy()
    assert np.array_equal(np.sort(od), np.arange(od.size)) and np.all(od[:wl.NB] >= wl.NB)   # head 1 first
    rp, cl = rowptr.cpu().numpy(), cols.cpu().numpy()
    for h in range(wl.H):
        c = {key: val[0, h] for key, val in x.items()}
        idx_h = oracle.estimate_topk(np64(c["q_lr"]), np64(c["k_lr"]), 64, ks[h])
        lists = _csr_lists(rp, cl, 0, h, wl.H, wl.NB)
        assert all(np.array_equal(lists[b], idx_h[b]) for b in range(wl.NB))
        ro, rl = oracle.sparse_attn_fwd(c["q"], c["k"], c["v"], idx_h, 64)
        assert_close(f"O[h{h}]", o[0, h], ro)
        assert_close(f"LSE[h{h}]", lse[0, h], rl, max_abs=LSE_MAX_ABS)
        rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], idx_h, 64)
        assert_close(f"dQ[h{h}]", dq[0, h], rdq)
        assert_close(f"dK[h{h}]", dk[0, h], rdk)
        assert_close(f"dV[h{h}]", dv[0, h], rdv)
