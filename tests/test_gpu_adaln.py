"""GPU parity of the fused AdaLN kernels (C ABI) against the fp64 oracle.

AdaptiveLoad page, technical summary section 2B: LayerNorm + modulation in one launch, and a
backward whose modulation gradients reduce over the sequence in (D tile, N tile) blocks.

Tolerance, from the arithmetic.  y and dx are bf16 roundings of fp32 results: the rounding
alone moves a value by up to 2^-8 of its magnitude (half an ulp at 8 significant bits), and
the fp32 statistics and products before it are accurate to far better than 2^-12 of the
magnitudes of the terms that make up the value.  Per element
    |got - ref| <= 2^-8 |ref| + 2^-12 * mag + 1e-6,
mag = |xhat (1 + scale)| + |shift| for y and rstd (|g| + |mean g| + |xhat mean(g xhat)|) for dx.
d_scale and d_shift are fp32 sums over the tokens: |got - ref| <= 2^-12 * sum_n |term| + 1e-6.
Every tensor also meets rel-L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_sparse_attention_estimate_gb300 import dsv_adaln_bwd, dsv_adaln_fwd
from dynamic_sparse_attention_estimate_gb300.inputs import ADALN_WORKLOADS, make_adaln_inputs
from tests.gpu_helpers import need_gpu, np64

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2


def _rel_l2(got, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got - ref)


def _bound_check(name, got, ref, mag, rel_mag=2.0 ** -12):
    excess = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + rel_mag * mag + 1e-6)
    worst = float(excess.max())
    r = _rel_l2(got, ref)
    assert worst <= 0 and r <= REL_L2, f"{name}: bound exceeded by {worst:.3e}, rel-L2 {r:.3e}"


def _magnitudes(x, scale, shift, dy, eps):
    """Per-element magnitudes of the terms of y and dx (fp64, from the bf16 inputs)."""
    x, scale, shift, dy = (np64(t) for t in (x, scale, shift, dy))
    mean = x.mean(-1, keepdims=True)
    rstd = 1.0 / np.sqrt(((x - mean) ** 2).mean(-1, keepdims=True) + eps)
    xhat = (x - mean) * rstd
    g = dy * (1.0 + scale[:, None, :])
    y_mag = np.abs(xhat * (1.0 + scale[:, None, :])) + np.abs(shift[:, None, :])
    dx_mag = rstd * (np.abs(g) + np.abs(g.mean(-1, keepdims=True)) + np.abs(xhat * (g * xhat).mean(-1, keepdims=True)))
    return y_mag, dx_mag, np.abs(dy * xhat).sum(1), np.abs(dy).sum(1)


def _check_all(inp, y, dx, ds, db, eps, rows=None):
    """Compare y / dx (on `rows` of sample 0 if given, else everything) and d_scale / d_shift."""
    x, scale, shift, dy = inp["x"], inp["scale"], inp["shift"], inp["dy"]
    if rows is None:
        xs, dys, ys, dxs = x, dy, y, dx
    else:
        xs, dys = x[:, rows], dy[:, rows]
        ys, dxs = y[:, rows], dx[:, rows]
    y_ref = oracle.adaln_fwd(xs, scale, shift, eps)
    dx_ref = oracle.adaln_bwd(xs, scale, dys, eps)[0]
    y_mag, dx_mag, _, _ = _magnitudes(xs, scale, shift, dys, eps)
    _bound_check("y", np64(ys), y_ref, y_mag)
    _bound_check("dx", np64(dxs), dx_ref, dx_mag)
    # modulation gradients: the oracle over row chunks, summed (the sums are over the tokens)
    N = x.shape[1]
    ds_ref = np.zeros(scale.shape)
    db_ref = np.zeros(scale.shape)
    ds_mag = np.zeros(scale.shape)
    db_mag = np.zeros(scale.shape)
    for a in range(0, N, 2048):
        _, s_, b_ = oracle.adaln_bwd(x[:, a:a + 2048], scale, dy[:, a:a + 2048], eps)
        ds_ref += s_
        db_ref += b_
        _, _, ms, mb = _magnitudes(x[:, a:a + 2048], scale, shift, dy[:, a:a + 2048], eps)
        ds_mag += ms
        db_mag += mb
    for name, got, ref, mag in (("d_scale", ds, ds_ref, ds_mag), ("d_shift", db, db_ref, db_mag)):
        g = np64(got)
        excess = np.abs(g - ref) - (2.0 ** -12 * mag + 1e-6)
        assert float(excess.max()) <= 0 and _rel_l2(g, ref) <= REL_L2, f"{name}: bound exceeded by {excess.max():.3e}"


def _run(inp, eps, dev):
    g = {k: v.to(dev) for k, v in inp.items()}
    y = dsv_adaln_fwd(g["x"], g["scale"], g["shift"], eps)
    dx, ds, db = dsv_adaln_bwd(g["x"], g["scale"], g["dy"], eps)
    torch.cuda.synchronize()
    return y, dx, ds, db


# (B, N, D): warps per row W = 1, 2, 4, 8 and 1..4 vectors per lane, ragged token tails,
# partial slabs (D = 1152: 144 vectors over 2 warps; D = 24: 3 vectors), one token, D = 8
@pytest.mark.parametrize("B,N,D", [(1, 1, 8), (1, 40, 24), (2, 37, 64), (1, 300, 768), (3, 129, 1152),
                                   (2, 65, 3072), (1, 19, 8192), (2, 1000, 256)])
def test_adaln_matches_oracle(B, N, D):
    dev = need_gpu()
    inp = make_adaln_inputs(B, N, D, seed=B * 1000 + D)
    y, dx, ds, db = _run(inp, 1e-6, dev)
    _check_all(inp, y, dx, ds, db, 1e-6)


@pytest.mark.parametrize("name", sorted(ADALN_WORKLOADS))
def test_adaln_full_size(name):
    """The bench workloads at full size: y / dx on 512 sampled tokens, d_scale / d_shift on all."""
    dev = need_gpu()
    B, N, D = ADALN_WORKLOADS[name]
    inp = make_adaln_inputs(B, N, D)
    y, dx, ds, db = _run(inp, 1e-6, dev)
    rows = np.sort(np.random.default_rng(5).choice(N, size=512, replace=False))
    _check_all(inp, y, dx, ds, db, 1e-6, rows=rows)


def test_adaln_large_eps_and_zero_eps():
    dev = need_gpu()
    inp = make_adaln_inputs(2, 77, 512, seed=3)
    for eps in (0.0, 0.25):
        y, dx, ds, db = _run(inp, eps, dev)
        _check_all(inp, y, dx, ds, db, eps)


def test_adaln_constant_rows_give_the_shift():
    """A constant token has zero variance: its normalised row is 0, so y is exactly the shift."""
    dev = need_gpu()
    inp = make_adaln_inputs(2, 50, 192, seed=4)
    inp["x"][0, 7] = 3.0
    inp["x"][1, 0] = -1.5
    inp["x"][1, 49] = 0.0
    y, dx, ds, db = _run(inp, 1e-6, dev)
    assert torch.equal(y[0, 7].cpu(), inp["shift"][0])
    assert torch.equal(y[1, 0].cpu(), inp["shift"][1])
    assert torch.equal(y[1, 49].cpu(), inp["shift"][1])
    _check_all(inp, y, dx, ds, db, 1e-6)


def test_adaln_deterministic():
    dev = need_gpu()
    B, N, D = ADALN_WORKLOADS["short"]
    g = {k: v.to(dev) for k, v in make_adaln_inputs(B, N, D).items()}
    a = dsv_adaln_bwd(g["x"], g["scale"], g["dy"])
    b = dsv_adaln_bwd(g["x"], g["scale"], g["dy"])
    ya = dsv_adaln_fwd(g["x"], g["scale"], g["shift"])
    yb = dsv_adaln_fwd(g["x"], g["scale"], g["shift"])
    torch.cuda.synchronize()
    assert torch.equal(ya, yb)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
