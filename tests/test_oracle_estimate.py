"""Pins for the oracle's estimate + top-k (CPU only).

The DSV pages print no worked example, so the selection is pinned by:
  * a hand-worked fixture (tests/golden/topk_hand.json),
  * brute force over every k-subset on tiny inputs (the unique subset satisfying the
    top-k-with-lower-index-tie-break conditions),
  * linearity of the block estimate: the block logit equals the sum of the per-token
    low-rank logits over the block (a different order of the same arithmetic),
  * selection invariants on larger random inputs.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import block_representatives, block_scores, estimate_topk, topk_select

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _is_topk_with_low_tiebreak(scores_row, subset):
    sel = set(subset)
    if len(sel) != len(subset):
        return False
    inside = [scores_row[j] for j in sel]
    outside = [j for j in range(len(scores_row)) if j not in sel]
    if not outside:
        return True
    lo = min(inside)
    hi = max(scores_row[j] for j in outside)
    if lo < hi:
        return False
    # at the boundary value every selected key must precede every unselected one
    if lo == hi:
        sel_at = [j for j in sel if scores_row[j] == lo]
        out_at = [j for j in outside if scores_row[j] == lo]
        if max(sel_at) > min(out_at):
            return False
    return True


def test_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "topk_hand.json")))
    q_lr = np.array(g["q_lr"], dtype=np.float64)
    k_lr = np.array(g["k_lr"], dtype=np.float64)
    q_hat = block_representatives(q_lr, g["block"])
    np.testing.assert_array_equal(q_hat, np.array(g["q_hat"]))
    np.testing.assert_array_equal(block_scores(q_hat, k_lr), np.array(g["scores"]))
    for k, want in g["idx"].items():
        got = estimate_topk(q_lr, k_lr, g["block"], int(k))
        np.testing.assert_array_equal(got, np.array(want, dtype=np.int32))


@pytest.mark.parametrize("seed", range(12))
def test_topk_equals_brute_force_subset(seed):
    rng = np.random.default_rng(seed)
    n = 9
    k = int(rng.integers(1, n))
    scores = rng.integers(-2, 3, size=(3, n)).astype(np.float64)  # small range -> many ties
    got = topk_select(scores, k)
    for row in range(scores.shape[0]):
        valid = [c for c in itertools.combinations(range(n), k) if _is_topk_with_low_tiebreak(scores[row], c)]
        assert len(valid) == 1, "the conditions must single out exactly one subset"
        assert list(got[row]) == sorted(valid[0])


def test_topk_invariants_random():
    rng = np.random.default_rng(7)
    for n, k in [(64, 1), (64, 64), (300, 37), (1000, 100)]:
        scores = rng.integers(-20, 21, size=(5, n)).astype(np.float64)
        idx = topk_select(scores, k)
        for row in range(scores.shape[0]):
            sel = idx[row]
            assert sel.shape == (k,)
            assert np.all(np.diff(sel) > 0), "ascending and distinct"
            assert sel.min() >= 0 and sel.max() < n
            assert _is_topk_with_low_tiebreak(scores[row], list(sel))


def test_topk_all_equal_scores_take_lowest_indices():
    scores = np.zeros((2, 50))
    np.testing.assert_array_equal(topk_select(scores, 7), np.tile(np.arange(7), (2, 1)))


def test_topk_full_density_is_arange():
    rng = np.random.default_rng(3)
    scores = rng.normal(size=(4, 33))
    np.testing.assert_array_equal(topk_select(scores, 33), np.tile(np.arange(33), (4, 1)))


def test_block_estimate_linearity():
    """Sum of per-token low-rank logits over a block == block representative logit."""
    rng = np.random.default_rng(11)
    block, nb, r, n_keys = 8, 5, 4, 23
    q_lr = rng.integers(-4, 5, size=(block * nb, r)).astype(np.float64)
    k_lr = rng.integers(-4, 5, size=(n_keys, r)).astype(np.float64)
    per_token = np.einsum("ic,jc->ij", q_lr, k_lr)
    summed = np.add.reduceat(per_token, np.arange(0, block * nb, block), axis=0)
    np.testing.assert_array_equal(block_scores(block_representatives(q_lr, block), k_lr), summed)


def test_block_representative_one_hot():
    """A block whose rows are unit vectors e_c counts how often each channel appears."""
    block, r = 6, 3
    rows = [0, 2, 2, 1, 2, 0]
    q_lr = np.eye(r)[rows]
    np.testing.assert_array_equal(block_representatives(q_lr, block)[0], [2, 1, 3])


def test_estimate_sampled_blocks_match_full():
    rng = np.random.default_rng(5)
    q_lr = rng.integers(-4, 5, size=(64 * 6, 16)).astype(np.float64)
    k_lr = rng.integers(-4, 5, size=(64 * 6, 16)).astype(np.float64)
    full = estimate_topk(q_lr, k_lr, 64, 40)
    part = estimate_topk(q_lr, k_lr, 64, 40, blocks=[4, 1])
    np.testing.assert_array_equal(part, full[[4, 1]])
