"""GPU parity at the large video shapes (full N, d, r, k; a subset of heads), on outputs the
oracle can compute one block at a time: selection on sampled blocks (every block for
the mid clip), O/LSE on sampled blocks, and the backward with dO zeroed outside the
sampled blocks (then only those blocks contribute to dK/dV, exactly).
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_sparse_attention_estimate_gb300 import dsv_estimate_topk, dsv_sparse_attn_bwd, dsv_sparse_attn_fwd
from dynamic_sparse_attention_estimate_gb300.binding import dsv_last_device_status
from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, make_inputs, sample_blocks

from gpu_helpers import LSE_MAX_ABS, assert_close, check_idx_invariants, need_gpu, np64

pytestmark = pytest.mark.gpu


def _sampled_check(wl, heads, n_sel_blocks, n_attn_blocks, all_blocks_selection=False):
    dev = need_gpu()
    x = make_inputs(wl, heads=heads)
    g = {k: v.to(dev) for k, v in x.items()}
    idx = dsv_estimate_topk(g["q_lr"], g["k_lr"], wl.k)
    o, lse = dsv_sparse_attn_fwd(g["q"], g["k"], g["v"], idx)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    check_idx_invariants(idx, wl.N)
    sel_blocks = np.arange(wl.NB) if all_blocks_selection else sample_blocks(wl.NB, n_sel_blocks, seed=1)
    attn_blocks = sample_blocks(wl.NB, n_attn_blocks, seed=2)
    mask = torch.zeros(wl.N, dtype=torch.bool)
    for b in attn_blocks:
        mask[b * 64:(b + 1) * 64] = True
    do_m = g["do"] * mask.to(dev)[None, None, :, None]
    dq, dk, dv = dsv_sparse_attn_bwd(do_m, g["q"], g["k"], g["v"], o, lse, idx)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    rows = mask.numpy()
    for hi in range(len(heads)):
        c = {key: val[0, hi] for key, val in x.items()}
        want = oracle.estimate_topk(c["q_lr"], c["k_lr"], 64, wl.k, blocks=sel_blocks)
        got = idx[0, hi][torch.from_numpy(sel_blocks).to(dev)].cpu().numpy()
        assert np.array_equal(got, want), f"head {heads[hi]}: selection differs"
        idx_h = idx[0, hi].cpu().numpy()
        ro, rl = oracle.sparse_attn_fwd(c["q"], c["k"], c["v"], idx_h, 64, blocks=attn_blocks)
        assert_close("O sampled", np64(o[0, hi])[rows], ro[rows])
        assert_close("LSE sampled", np64(lse[0, hi])[rows], rl[rows], max_abs=LSE_MAX_ABS)
        rdq, rdk, rdv = oracle.sparse_attn_bwd(c["do"], c["q"], c["k"], c["v"], idx_h, 64, blocks=attn_blocks,
                                               o=ro, lse=rl)
        assert_close("dQ sampled", np64(dq[0, hi])[rows], rdq[rows])
        assert_close("dK", dk[0, hi], rdk)
        assert_close("dV", dv[0, hi], rdv)
    return g, idx, o


def test_mid_clip_planted_locality():
    wl = WORKLOADS["mid"]
    _sampled_check(wl, heads=[0, wl.H - 1], n_sel_blocks=0, n_attn_blocks=24, all_blocks_selection=True)


@pytest.mark.parametrize("density", [0.05, 0.10, 0.20, 1.00])
def test_density_sweep(density):
    wl = WORKLOADS["sweep"].with_density(density)
    g, idx, o = _sampled_check(wl, heads=[0, 1], n_sel_blocks=48, n_attn_blocks=8 if density < 1 else 4)
    if density == 1.0:
        ref = torch.nn.functional.scaled_dot_product_attention(g["q"], g["k"], g["v"])
        assert_close("O vs dense SDPA", o, np64(ref))


def test_long_video_one_call_of_four_heads():
    wl = WORKLOADS["long"]
    _sampled_check(wl, heads=[0, 1, 2, 3], n_sel_blocks=64, n_attn_blocks=64)

