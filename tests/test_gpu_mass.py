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


def _select(g, tau, mass):
    k_row, rowptr = dsv_estimate_mass_k(g["q_lr"], g["k_lr"], tau, mass)
    cols = dsv_estimate_topk_csr(g["q_lr"], g["k_lr"], k_row, rowptr)
    torch.cuda.synchronize()
    assert dsv_last_device_status() == 0
    return k_row.cpu().numpy(), rowptr.cpu().numpy(), cols.cpu().numpy()


def _check_head(x, b, h, k_row, rowptr, cols, tau, mass):
    tau_log2, mass_num = mass_parameters(tau, mass)
    s = oracle.block_scores(oracle.block_representatives(np64(x["q_lr"][b, h]), 64), np64(x["k_lr"][b, h]))
    want_k = oracle.mass_k(s, tau_log2, mass_num)
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
