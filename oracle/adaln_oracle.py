"""Plain, slow, fp64 CPU oracle of the fused AdaLN (LayerNorm + modulation) operator.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline leg may import this module.  It shares no code with the CUDA path and
imports nothing from the package.

What it computes follows the AdaptiveLoad page ("AdaptiveLoad: Towards Efficient Video
Diffusion Transformer Training", technical summary, section 2B "fused LayerNorm-Modulate
CUDA kernel"):

* forward: per token, the mean and the variance of its D features (two reductions),
  then the normalised row is modulated by the sample's (scale, shift) vectors in a
  third pass over D;
* backward: the gradient of x, and the gradients of the modulation vectors, which are
  sums over the sequence dimension N (the reduction the page reorganises into
  (D tile, N tile) blocks so that reads stay coalesced).

Readings where the page is silent:
  1. modulation is the DiT form y = LN(x) * (1 + scale) + shift, with (scale, shift)
     one D-vector per sample, broadcast over that sample's tokens;
  2. LN has no learned affine of its own; the variance is the biased one (divided
     by D) and eps is added inside the square root: rstd = 1 / sqrt(var + eps);
  3. the backward recomputes mean and rstd from x (the statistics are not saved
     between the passes: the page keeps them in registers to cut activation memory);
  4. gradients are returned for x, scale and shift.

Every step is written the obvious way with numpy fp64; no blocking or fusion.
Shapes: x, dy [B, N, D]; scale, shift [B, D].
"""
from __future__ import annotations

from typing import Tuple

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def row_stats(x, eps: float) -> Tuple[np.ndarray, np.ndarray]:
    """(mean [B, N], rstd [B, N]): the first two passes over each token's D features."""
    x = _f64(x)
    mean = x.mean(axis=-1)
    var = ((x - mean[..., None]) ** 2).mean(axis=-1)
    return mean, 1.0 / np.sqrt(var + eps)


def adaln_fwd(x, scale, shift, eps: float = 1e-6) -> np.ndarray:
    """y [B, N, D] = (x - mean) * rstd * (1 + scale[b]) + shift[b]."""
    x, scale, shift = _f64(x), _f64(scale), _f64(shift)
    mean, rstd = row_stats(x, eps)
    xhat = (x - mean[..., None]) * rstd[..., None]
    return xhat * (1.0 + scale[:, None, :]) + shift[:, None, :]


def adaln_bwd(x, scale, dy, eps: float = 1e-6) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(dx [B, N, D], d_scale [B, D], d_shift [B, D]) for the loss gradient dy.

    With xhat = (x - mean) * rstd and g = dy * (1 + scale):
      d_shift[b, d] = sum_n dy[b, n, d]
      d_scale[b, d] = sum_n dy[b, n, d] * xhat[b, n, d]
      dx = rstd * (g - mean_D(g) - xhat * mean_D(g * xhat))
    (the chain rule through the per-row mean and rstd).
    """
    x, scale, dy = _f64(x), _f64(scale), _f64(dy)
    mean, rstd = row_stats(x, eps)
    xhat = (x - mean[..., None]) * rstd[..., None]
    d_shift = dy.sum(axis=1)
    d_scale = (dy * xhat).sum(axis=1)
    g = dy * (1.0 + scale[:, None, :])
    mg = g.mean(axis=-1, keepdims=True)
    mgx = (g * xhat).mean(axis=-1, keepdims=True)
    dx = rstd[..., None] * (g - mg - xhat * mgx)
    return dx, d_scale, d_shift
