"""Pins of the fused AdaLN oracle (CPU only).

AdaptiveLoad page, technical summary section 2B: LayerNorm statistics per token, then the
modulation of the normalised row; in the backward, the gradient of x and the modulation
gradients, which reduce over the sequence.  The pins tie the oracle to an independent
library (torch fp64 layer_norm and autograd), to finite differences, and to invariances of
the true function (a per-row constant added to x changes nothing; at eps = 0 neither does a
positive per-row factor; y is linear in scale and shift), and a planted mistake anywhere in
the oracle fails at least one of them.
"""
import types

import numpy as np
import pytest
import torch

import oracle.adaln_oracle as real

SRC = open(real.__file__).read()


def _mutant(old, new):
    assert SRC.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant_adaln")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant_adaln", "exec"), mod.__dict__)
    return mod


def _case(B=2, N=5, D=12, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(B, N, D)) * rng.uniform(0.5, 3.0, size=(B, N, 1)) + rng.normal(size=(B, N, 1))
    scale = rng.normal(size=(B, D)) * 0.5
    shift = rng.normal(size=(B, D))
    dy = rng.normal(size=(B, N, D))
    return x, scale, shift, dy


def _torch_ref(x, scale, shift, dy, eps):
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    st = torch.tensor(scale, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(shift, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.layer_norm(xt, (x.shape[-1],), eps=eps) * (1 + st[:, None, :]) + bt[:, None, :]
    y.backward(torch.tensor(dy, dtype=torch.float64))
    return y.detach().numpy(), xt.grad.numpy(), st.grad.numpy(), bt.grad.numpy()


# ---------------------------------------------------------------- the pins, as predicates on a module

def _torch_fwd_ok(m):
    for eps in (1e-6, 1e-2):
        x, s, b, dy = _case()
        y_ref = _torch_ref(x, s, b, dy, eps)[0]
        if not np.allclose(m.adaln_fwd(x, s, b, eps), y_ref, rtol=1e-12, atol=1e-12):
            return False
    return True


def _torch_bwd_ok(m):
    for eps in (1e-6, 1e-2):
        x, s, b, dy = _case(seed=1)
        _, dx_ref, ds_ref, db_ref = _torch_ref(x, s, b, dy, eps)
        dx, ds, db = m.adaln_bwd(x, s, dy, eps)
        if not (np.allclose(dx, dx_ref, rtol=1e-10, atol=1e-12) and np.allclose(ds, ds_ref, rtol=1e-10, atol=1e-12)
                and np.allclose(db, db_ref, rtol=1e-10, atol=1e-12)):
            return False
    return True


def _finite_difference_ok(m):
    eps, h = 1e-3, 1e-6
    x, s, b, dy = _case(B=2, N=3, D=5, seed=2)
    loss = lambda x_, s_, b_: float((m.adaln_fwd(x_, s_, b_, eps) * dy).sum())
    dx, ds, db = m.adaln_bwd(x, s, dy, eps)
    for arr, grad, which in ((x, dx, 0), (s, ds, 1), (b, db, 2)):
        for flat in range(arr.size):
            e = np.zeros(arr.size)
            e[flat] = h
            e = e.reshape(arr.shape)
            args_p, args_m = [x, s, b], [x, s, b]
            args_p[which] = arr + e
            args_m[which] = arr - e
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            if abs(fd - grad.reshape(-1)[flat]) > 1e-6 * max(1.0, abs(fd)):
                return False
    return True


def _invariances_ok(m):
    x, s, b, dy = _case(seed=3)
    c = np.random.default_rng(4).normal(size=x.shape[:2] + (1,)) * 5
    a = np.random.default_rng(5).uniform(0.2, 4.0, size=x.shape[:2] + (1,))
    for eps in (1e-6, 0.5):
        if not np.allclose(m.adaln_fwd(x + c, s, b, eps), m.adaln_fwd(x, s, b, eps), rtol=1e-9, atol=1e-9):
            return False
    if not np.allclose(m.adaln_fwd(x * a, s, b, 0.0), m.adaln_fwd(x, s, b, 0.0), rtol=1e-9, atol=1e-9):
        return False
    # the gradient of a function invariant to x + c*1 sums to 0 per row (any eps); at eps = 0
    # the function is also invariant to x * a, so the gradient is orthogonal to x - mean
    for eps in (1e-6, 0.5):
        dx = m.adaln_bwd(x, s, dy, eps)[0]
        if np.max(np.abs(dx.sum(-1))) > 1e-9 * np.abs(dx).sum(-1).max():
            return False
    dx = m.adaln_bwd(x, s, dy, 0.0)[0]
    xc = x - x.mean(-1, keepdims=True)
    return np.max(np.abs((dx * xc).sum(-1))) < 1e-9 * np.abs(dx * xc).sum(-1).max()


def _constant_rows_ok(m):
    # a constant row has zero variance: its normalised row is 0 and y is the shift
    x = np.full((2, 3, 8), 2.5)
    x[1] = -7.0
    s, b = np.random.default_rng(6).normal(size=(2, 8)), np.random.default_rng(7).normal(size=(2, 8))
    return np.array_equal(m.adaln_fwd(x, s, b, 1e-6), np.broadcast_to(b[:, None, :], x.shape))


def _normalised_moments_ok(m):
    # scale = shift = 0: each output row has mean 0 and mean square var / (var + eps)
    x, _, _, _ = _case(seed=8)
    z = np.zeros((x.shape[0], x.shape[-1]))
    for eps in (1e-6, 0.3):
        y = m.adaln_fwd(x, z, z, eps)
        var = x.var(-1)
        if not (np.allclose(y.mean(-1), 0, atol=1e-12) and np.allclose((y ** 2).mean(-1), var / (var + eps),
                                                                       rtol=1e-12)):
            return False
    return True


def _linear_in_modulation_ok(m):
    # y is affine in (scale, shift): the exact directional change along e_d is dy . xhat (scale)
    # and dy (shift), summed over the tokens -- which is what d_scale and d_shift must be
    x, s, b, dy = _case(seed=9)
    eps, t = 1e-6, 0.75
    dx, ds, db = m.adaln_bwd(x, s, dy, eps)
    base = (m.adaln_fwd(x, s, b, eps) * dy).sum()
    for bb in range(s.shape[0]):
        for d in range(s.shape[1]):
            s2, b2 = s.copy(), b.copy()
            s2[bb, d] += t
            b2[bb, d] += t
            if abs(((m.adaln_fwd(x, s2, b, eps) * dy).sum() - base) / t - ds[bb, d]) > 1e-9:
                return False
            if abs(((m.adaln_fwd(x, s, b2, eps) * dy).sum() - base) / t - db[bb, d]) > 1e-9:
                return False
    return True


PINS = [_torch_fwd_ok, _torch_bwd_ok, _finite_difference_ok, _invariances_ok, _constant_rows_ok,
        _normalised_moments_ok, _linear_in_modulation_ok]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_meets_pin(pin):
    assert pin(real)


MUTANTS = {
    "unbiased variance": ("var = ((x - mean[..., None]) ** 2).mean(axis=-1)",
                          "var = ((x - mean[..., None]) ** 2).sum(axis=-1) / (x.shape[-1] - 1)"),
    "eps outside the root": ("1.0 / np.sqrt(var + eps)", "1.0 / (np.sqrt(var) + eps)"),
    "modulation without the one": ("return xhat * (1.0 + scale[:, None, :])", "return xhat * scale[:, None, :]"),
    "shift on the wrong side": ("return xhat * (1.0 + scale[:, None, :]) + shift[:, None, :]",
                                "return (xhat + shift[:, None, :]) * (1.0 + scale[:, None, :])"),
    "dropped projection term": ("dx = rstd[..., None] * (g - mg - xhat * mgx)", "dx = rstd[..., None] * (g - mg)"),
    "dropped mean term": ("dx = rstd[..., None] * (g - mg - xhat * mgx)", "dx = rstd[..., None] * (g - xhat * mgx)"),
    "dx without rstd": ("dx = rstd[..., None] * (g - mg - xhat * mgx)", "dx = (g - mg - xhat * mgx)"),
    "projection on dy, not g": ("mgx = (g * xhat).mean(axis=-1, keepdims=True)",
                                "mgx = (dy * xhat).mean(axis=-1, keepdims=True)"),
    "d_scale without rstd": ("d_scale = (dy * xhat).sum(axis=1)",
                             "d_scale = (dy * (x - mean[..., None])).sum(axis=1)"),
    "d_shift over features": ("d_shift = dy.sum(axis=1)", "d_shift = np.broadcast_to(dy.sum(axis=2).sum(axis=1, keepdims=True), (dy.shape[0], dy.shape[2]))"),
    "g without the one": ("g = dy * (1.0 + scale[:, None, :])", "g = dy * scale[:, None, :]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = _mutant(*MUTANTS[name])
    assert not all(pin(m) for pin in PINS), name
