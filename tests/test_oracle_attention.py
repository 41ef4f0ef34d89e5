"""Pins for the oracle's sparse attention forward and backward (CPU only).

Independent references:
  * torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU, at density
    100 % (the dense special case) and with a -inf mask outside the selected set;
  * torch fp64 autograd of that masked dense form for the backward;
  * central finite differences of sum(dO * O) through the oracle's own forward;
  * closed forms: sum_j dV_j = sum_i dO_i (rows of P sum to one), sum_j dK_j = 0
    (each row of dS sums to zero), zero gradient for keys no block selected;
  * a hand-worked fixture (tests/golden/attn_hand.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import sparse_attn_bwd, sparse_attn_fwd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, n=256, d=16, block=32, k=40):
    rng = np.random.default_rng(seed)
    q, kk, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    nb = n // block
    idx = np.stack([np.sort(rng.choice(n, size=k, replace=False)) for _ in range(nb)]).astype(np.int32)
    return q, kk, v, do, idx


def _mask_from_idx(idx, n, block):
    mask = torch.full((n, n), float("-inf"), dtype=torch.float64)
    for b in range(idx.shape[0]):
        mask[b * block:(b + 1) * block, torch.from_numpy(idx[b].astype(np.int64))] = 0.0
    return mask


def _sdpa(q, k, v, mask, scale):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, scale=scale)[0, 0]


def test_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "attn_hand.json")))
    arr = lambda key: np.array(g[key], dtype=np.float64)
    q, k, v, do = arr("q"), arr("k"), arr("v"), arr("do")
    idx = np.array(g["idx"], dtype=np.int32)
    o, lse = sparse_attn_fwd(q, k, v, idx, g["block"], g["scale"], blocks=[0])
    np.testing.assert_allclose(o[:2], arr("O_block0"), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:2], arr("LSE_block0"), rtol=0, atol=1e-14)
    dq, dk, dv = sparse_attn_bwd(do, q, k, v, idx, g["block"], g["scale"], blocks=[0])
    np.testing.assert_allclose(dq[0], g["dQ_row0"], atol=1e-14)
    for key, want in g["dK"].items():
        np.testing.assert_allclose(dk[int(key)], want, atol=1e-14)
    for key, want in g["dV"].items():
        np.testing.assert_allclose(dv[int(key)], want, atol=1e-14)


@pytest.mark.parametrize("seed", [0, 1])
def test_full_density_equals_dense_sdpa(seed):
    n, d, block = 192, 32, 64
    q, k, v, _, _ = _rand_case(seed, n, d, block, 1)
    idx = np.tile(np.arange(n, dtype=np.int32), (n // block, 1))
    scale = 1 / math.sqrt(d)
    o, lse = sparse_attn_fwd(q, k, v, idx, block, scale)
    ref = _sdpa(q, k, v, None, scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(scale * torch.from_numpy(q) @ torch.from_numpy(k).T, dim=1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sparse_equals_dense_with_minus_inf_mask(seed):
    n, d, block, k = 256, 16, 32, 40
    q, kk, v, _, idx = _rand_case(seed, n, d, block, k)
    scale = 0.37
    o, lse = sparse_attn_fwd(q, kk, v, idx, block, scale)
    mask = _mask_from_idx(idx, n, block)
    np.testing.assert_allclose(o, _sdpa(q, kk, v, mask, scale).numpy(), rtol=1e-12, atol=1e-12)
    logits = scale * torch.from_numpy(q) @ torch.from_numpy(kk).T + mask
    np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=1).numpy(), rtol=1e-12, atol=1e-12)


def test_probabilities_sum_to_one_and_output_is_convex():
    q, k, v, _, idx = _rand_case(4)
    block = 32
    scale = 0.25
    o, lse = sparse_attn_fwd(q, k, v, idx, block, scale)
    for b in range(idx.shape[0]):
        rows = slice(b * block, (b + 1) * block)
        p = np.exp(scale * q[rows] @ k[idx[b]].T - lse[rows][:, None])
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
        vsel = v[idx[b]]
        assert np.all(o[rows] <= vsel.max(axis=0) + 1e-12) and np.all(o[rows] >= vsel.min(axis=0) - 1e-12)


def test_permuting_idx_rows_changes_nothing():
    q, k, v, do, idx = _rand_case(5)
    rng = np.random.default_rng(9)
    shuffled = np.stack([rng.permutation(row) for row in idx])
    o1, l1 = sparse_attn_fwd(q, k, v, idx, 32)
    o2, l2 = sparse_attn_fwd(q, k, v, shuffled, 32)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    g1 = sparse_attn_bwd(do, q, k, v, idx, 32)
    g2 = sparse_attn_bwd(do, q, k, v, shuffled, 32)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_equals_torch_autograd_of_masked_dense(seed):
    n, d, block, k = 128, 16, 32, 24
    q, kk, v, do, idx = _rand_case(seed, n, d, block, k)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = sparse_attn_bwd(do, q, kk, v, idx, block, scale)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, kk, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=_mask_from_idx(idx, n, block), scale=scale)[0, 0]
    (out * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_central_finite_differences():
    n, d, block, k = 64, 8, 16, 12
    q, kk, v, do, idx = _rand_case(3, n, d, block, k)
    scale = 0.5
    dq, dk, dv = sparse_attn_bwd(do, q, kk, v, idx, block, scale)

    def loss(qq, kx, vx):
        o, _ = sparse_attn_fwd(qq, kx, vx, idx, block, scale)
        return float((o * do).sum())

    h = 1e-6
    rng = np.random.default_rng(1)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(6):
            i, c = int(rng.integers(n)), int(rng.integers(d))
            args_p = [q.copy(), kk.copy(), v.copy()]
            args_m = [q.copy(), kk.copy(), v.copy()]
            args_p[which][i, c] += h
            args_m[which][i, c] -= h
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[i, c]) <= 1e-6 * max(1.0, abs(fd)), (which, i, c, fd, grad[i, c])


def test_backward_closed_forms_and_unselected_keys():
    n, d, block, k = 256, 16, 32, 20
    q, kk, v, do, idx = _rand_case(8, n, d, block, k)
    dq, dk, dv = sparse_attn_bwd(do, q, kk, v, idx, block, 0.3)
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-10)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-10)
    unselected = np.setdiff1d(np.arange(n), np.unique(idx))
    assert unselected.size > 0
    assert np.all(dk[unselected] == 0) and np.all(dv[unselected] == 0)


def test_sampled_blocks_equal_zeroed_dO_elsewhere():
    """Restricting the backward to some blocks == running it with dO = 0 outside them."""
    n, d, block, k = 256, 16, 32, 30
    q, kk, v, do, idx = _rand_case(6, n, d, block, k)
    blocks = [1, 6]
    masked = np.zeros_like(do)
    for b in blocks:
        masked[b * block:(b + 1) * block] = do[b * block:(b + 1) * block]
    full = sparse_attn_bwd(masked, q, kk, v, idx, block)
    part = sparse_attn_bwd(do, q, kk, v, idx, block, blocks=blocks)
    for a, b in zip(full, part):
        np.testing.assert_allclose(a, b, atol=1e-12)
