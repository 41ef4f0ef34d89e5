"""Pins of the oracle's mass-based adaptive k (CPU only).

DSV pages, German summary section 2A stage 2 and Spanish "Fase 2": the critical KV pairs are
those that make up ~90 % of the (estimated) attention score.  The oracle takes, per block,
the shortest (score desc, key asc) prefix whose integer weight reaches the mass target; the
weights come from a fixed fp32 exp2 recipe.  These pins tie the recipe to 2^x, the search to
its definition (sufficient and minimal), and both to closed forms.
"""
import math
import types

import numpy as np
import pytest

import oracle.dsv_oracle as real

SRC = open(real.__file__).read()
ONE = 1 << 24                      # weight of a key at the block maximum


def _mutant(old, new):
    assert SRC.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant_mass")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant_mass", "exec"), mod.__dict__)
    return mod


def _recipe_ok(m):
    x = -np.linspace(0.0, 29.99, 20001).astype(np.float32)
    got = m.exp2_recipe(x).astype(np.float64)
    return np.max(np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)) < 2e-5


def _equal_scores_ok(m):
    # N equal scores: every weight is 2^24, so k = ceil(target / 2^24) = ceil(N * mass)
    for n in (10, 64, 1000):
        s = np.full((1, n), 7.0)
        for num in (65536, 32768, 58982, 1):
            want = math.ceil(((n * ONE * num + 65535) >> 16) / ONE)
            if int(m.mass_k(s, 0.1, num)[0]) != want:
                return False
    return True


def _target_ok(m):
    # the target is the least integer t with t * 2^16 >= W * mass_num
    rng = np.random.default_rng(5)
    for _ in range(2000):
        w, num = int(rng.integers(1, 1 << 44)), int(rng.integers(1, 65537))
        t = m.mass_target(w, num)
        if not (t * 65536 >= w * num and (t - 1) * 65536 < w * num):
            return False
    return True


def _sufficient_and_minimal(m, scores, tau_log2, num):
    ks = m.mass_k(scores, tau_log2, num)
    for b in range(scores.shape[0]):
        order = np.lexsort((np.arange(scores.shape[1]), -scores[b]))
        w = [int(x) for x in m.mass_weights(scores[b], tau_log2)[order]]
        target = m.mass_target(sum(w), num)
        k = int(ks[b])
        if not (sum(w[:k]) >= target and sum(w[:k - 1]) < target):
            return False
    return True


def test_recipe_matches_exp2_and_is_exact_at_integers():
    assert _recipe_ok(real)
    x = -np.arange(0, 31, dtype=np.float32)
    assert np.array_equal(real.exp2_recipe(x), np.exp2(x))        # f = 0: the series gives 1 exactly


def test_weights_top_key_and_cutoff():
    s = np.array([5.0, 5.0, 3.0, -1e4])
    w = real.mass_weights(s, 1.0)
    assert w[0] == ONE and w[1] == ONE          # the maximum weighs 2^24
    assert w[2] == ONE // 4                     # 2^-2
    assert w[3] == 0                            # far below: no weight


def test_target_is_the_least_sufficient_integer():
    assert _target_ok(real)


def test_equal_scores_closed_form():
    assert _equal_scores_ok(real)


def test_dominant_key_alone():
    s = np.zeros((1, 300))
    s[0, 123] = 1e3
    assert int(real.mass_k(s, 1.0, 58982)[0]) == 1


def test_sufficient_and_minimal_on_random_rows():
    rng = np.random.default_rng(1)
    for tau in (0.02, 0.2, 1.5):
        s = rng.integers(-60, 60, size=(6, 257)).astype(np.float64)
        for num in (1, 32768, 58982, 65536):
            assert _sufficient_and_minimal(real, s, tau, num)


def test_k_grows_with_mass_and_ignores_key_order():
    rng = np.random.default_rng(2)
    s = rng.integers(-30, 30, size=(4, 500)).astype(np.float64)
    ks = [real.mass_k(s, 0.1, num) for num in (6554, 32768, 58982, 65536)]
    for a, b in zip(ks, ks[1:]):
        assert np.all(a <= b)
    perm = rng.permutation(500)
    assert np.array_equal(real.mass_k(s[:, perm], 0.1, 58982), ks[2])


def test_selection_is_the_top_k_of_each_block():
    rng = np.random.default_rng(3)
    n, r, block = 256, 16, 64
    q_lr = rng.integers(-4, 5, size=(n, r)).astype(np.float64)
    k_lr = rng.integers(-4, 5, size=(n, r)).astype(np.float64)
    ks, sel = real.estimate_mass_topk(q_lr, k_lr, block, 0.05, 58982)
    s = real.block_scores(real.block_representatives(q_lr, block), k_lr)
    for b in range(n // block):
        assert len(sel[b]) == ks[b]
        assert np.array_equal(sel[b], real.topk_select(s[b:b + 1], int(ks[b]))[0])


@pytest.mark.parametrize("old,new,pin", [
    ("p = np.float32(EXP2_TAYLOR[6]) * np.ones_like(f)", "p = np.float32(0.0) * np.ones_like(f)", _recipe_ok),
    ("p = (p + c).astype(np.float32)", "p = (p - c).astype(np.float32)", _recipe_ok),
    ("    n = np.floor(x).astype(np.float32)", "    n = np.ceil(x).astype(np.float32)", _recipe_ok),
    ("return (int(total) * int(mass_num) + 65535) >> 16", "return (int(total) * int(mass_num)) >> 16", lambda m: _target_ok(m)),
    ("out[b] = int(np.argmax(cum >= target)) + 1", "out[b] = int(np.argmax(cum > target)) + 1", _equal_scores_ok),
    ("order = np.lexsort((np.arange(scores.shape[1]), -scores[b]))",
     "order = np.lexsort((np.arange(scores.shape[1]), scores[b]))",
     lambda m: _sufficient_and_minimal(real, np.random.default_rng(4).integers(-40, 40, size=(3, 100)).astype(float), 0.3, 58982)
     and np.array_equal(m.mass_k(np.random.default_rng(4).integers(-40, 40, size=(3, 100)).astype(float), 0.3, 58982),
                        real.mass_k(np.random.default_rng(4).integers(-40, 40, size=(3, 100)).astype(float), 0.3, 58982))),
])
def test_mutants_are_rejected(old, new, pin):
    assert pin(real)
    assert not pin(_mutant(old, new))


def test_ragged_selection_attention_equals_masked_dense():
    # per-block key lists of different lengths: attention over them = dense attention with
    # -inf outside each block's list (torch fp64 SDPA, an independent library)
    import torch
    rng = np.random.default_rng(6)
    n, d, block = 192, 16, 64
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    sel = [np.sort(rng.choice(n, size=m, replace=False)).astype(np.int32) for m in (5, 64, 150)]
    mask = torch.full((n, n), float("-inf"), dtype=torch.float64)
    for b, s in enumerate(sel):
        mask[b * block:(b + 1) * block, torch.from_numpy(s.astype(np.int64))] = 0
    scale = 1 / math.sqrt(d)
    o, lse = real.sparse_attn_fwd(q, k, v, sel, block, scale)
    t = lambda a: torch.from_numpy(a)[None, None].requires_grad_(True)
    tq, tk, tv = t(q), t(k), t(v)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    assert np.allclose(o, ref[0, 0].detach().numpy(), atol=1e-10)
    ref.backward(torch.from_numpy(do)[None, None])
    dq, dk, dv = real.sparse_attn_bwd(do, q, k, v, sel, block, scale)
    for got, want in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.allclose(got, want.grad[0, 0].numpy(), atol=1e-9)


def test_sparse_dense_switch():
    # dense_num = 0: off; 65536: never (k <= N); otherwise k * 2^16 > dense_num * N -> N
    rng = np.random.default_rng(7)
    s = rng.integers(-20, 20, size=(8, 300)).astype(np.float64)
    base = real.mass_k(s, 0.05, 58982)
    assert np.array_equal(real.mass_k(s, 0.05, 58982, 0), base)
    assert np.array_equal(real.mass_k(s, 0.05, 58982, 65536), base)
    for num in (1, 9830, 32768):
        got = real.mass_k(s, 0.05, 58982, num)
        want = np.where(base.astype(np.int64) * 65536 > num * 300, 300, base)
        assert np.array_equal(got, want)
