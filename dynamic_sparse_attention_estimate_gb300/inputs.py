"""Seeded synthetic inputs for DSV's dynamic sparse 3D attention and the fused AdaLN operator.

This module only draws random numbers and lays tokens out; it holds none of the
method's arithmetic (no estimate, no selection, no attention). Both the CUDA path
and the CPU oracle consume what it produces, so it imports neither of them.

Workloads (the video-shaped shapes the DSV pages talk about: long 3D latents of
16k-520k tokens, per-head low-rank factors, about 10% of the keys kept):

  tiny   B=1 H=2  latent 4x16x16   -> N=1,024    d=64  r=16 k=128    raster blocks
  short  B=1 H=12 latent 16x32x32  -> N=16,384   d=64  r=16 k=1,638  4x4x4 cubes
  mid    B=1 H=24 latent 16x64x64  -> N=65,536   d=128 r=32 k=6,553  cubes, planted locality
  sweep  B=1 H=24 latent 32x64x64  -> N=131,072  d=128 r=32 k=5/10/20/100% of N
  long   B=1 H=24 latent 127x64x64 -> N=520,192  d=128 r=16 k=52,019 (4 heads per call)

Token order.  Tokens are generated in raster (t, h, w) order and then permuted to
"block-major" order, so that query block b covers rows [64 b, 64 b + 64).  A block is
a group of 3D-neighbouring tokens (DSV page 1, technical summary section 2B, "Query
Grouping": neighbouring tokens in space-time share critical keys).  The tiny workload
uses 64 consecutive raster tokens per block; the others use 4x4x4 cubes in
cube-raster order with raster order inside a cube; the long workload's last three
frames (127 = 4*31 + 3) use 1x8x8 tiles.

Random streams.  Every (batch, head) slice has its own torch CPU generator seeded
with ``seed + 7919 * (b * H + h)`` so that any head subset can be produced alone.
Within a slice the draw order is Q, K, V, dO, Q_lr, K_lr (the mid workload: Q, K0,
e, V, dO).  Q, K, V, dO are N(0, 1) rounded to bf16; integer low-rank factors are
uniform on the inclusive range [-lr_max, lr_max] and stored as bf16 (exact).  The
mid workload's random +-1 projection R is shared by Q, K and all heads and comes
from a generator seeded with ``seed + 104729``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import numpy as np
import torch

BLOCK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    latent: tuple  # (T, Hh, W)
    d: int
    r: int
    k: int
    block_shape: Optional[tuple]  # None -> consecutive raster tokens
    lr_max: int = 4
    planted_locality: bool = False
    heads_per_call: Optional[int] = None
    seed: int = 0

    @property
    def N(self) -> int:
        t, h, w = self.latent
        return t * h * w

    @property
    def NB(self) -> int:
        return self.N // BLOCK

    @property
    def density(self) -> float:
        return self.k / self.N

    def with_density(self, density: float) -> "Workload":
        """Same shapes with k = floor(density * N) (k from a density: the plainest reading)."""
        k = int(math.floor(density * self.N + 1e-9))
        return dataclasses.replace(self, k=max(1, min(self.N, k)))

    def with_heads(self, H: int) -> "Workload":
        return dataclasses.replace(self, H=H)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 2, (4, 16, 16), 64, 16, 128, None),
    "short": Workload("short", 1, 12, (16, 32, 32), 64, 16, 1638, (4, 4, 4)),
    "mid": Workload("mid", 1, 24, (16, 64, 64), 128, 32, 6553, (4, 4, 4),
                    lr_max=8, planted_locality=True),
    "sweep": Workload("sweep", 1, 24, (32, 64, 64), 128, 32, 13107, (4, 4, 4)),
    "long": Workload("long", 1, 24, (127, 64, 64), 128, 16, 52019, (4, 4, 4),
                     heads_per_call=4),
}
SWEEP_DENSITIES = (0.05, 0.10, 0.20, 1.00)


def block_major_permutation(latent: Sequence[int], block_shape: Optional[Sequence[int]]) -> np.ndarray:
    """perm[p] = raster index of the token stored at block-major position p."""
    T, Hh, W = latent
    raster = np.arange(T * Hh * W, dtype=np.int64).reshape(T, Hh, W)
    if block_shape is None:
        return raster.reshape(-1)
    bt, bh, bw = block_shape
    assert bt * bh * bw == BLOCK and Hh % bh == 0 and W % bw == 0
    parts = []
    t_cubes = (T // bt) * bt
    # cubes of bt x bh x bw, cube-raster order, raster inside each cube
    cube = raster[:t_cubes].reshape(T // bt, bt, Hh // bh, bh, W // bw, bw)
    parts.append(cube.transpose(0, 2, 4, 1, 3, 5).reshape(-1))
    if t_cubes < T:
        # leftover frames: 1 x 8 x 8 tiles (still 64 tokens per block)
        th, tw = 8, 8
        assert Hh % th == 0 and W % tw == 0
        rest = raster[t_cubes:].reshape(T - t_cubes, Hh // th, th, W // tw, tw)
        parts.append(rest.transpose(0, 1, 3, 2, 4).reshape(-1))
    perm = np.concatenate(parts)
    assert perm.size == T * Hh * W
    return perm


def _head_generator(wl: Workload, b: int, h: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed + 7919 * (b * wl.H + h))
    return g


def _normal_bf16(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _int_bf16(g: torch.Generator, shape, lim: int) -> torch.Tensor:
    return torch.randint(-lim, lim + 1, shape, generator=g, dtype=torch.int32).to(torch.bfloat16)


def projection_matrix(wl: Workload) -> torch.Tensor:
    """The mid workload's seeded +-1 matrix R of shape [d, r] (fp32)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed + 104729)
    bits = torch.randint(0, 2, (wl.d, wl.r), generator=g, dtype=torch.int32)
    return (bits * 2 - 1).to(torch.float32)


def _neighbourhood_of_token(latent, nb_shape=(4, 8, 8)) -> np.ndarray:
    """Raster token -> index of its 4x8x8 neighbourhood (mid workload's planted structure)."""
    T, Hh, W = latent
    t = np.arange(T)[:, None, None] // nb_shape[0]
    y = np.arange(Hh)[None, :, None] // nb_shape[1]
    x = np.arange(W)[None, None, :] // nb_shape[2]
    ny, nx = Hh // nb_shape[1], W // nb_shape[2]
    return ((t * ny + y) * nx + x).reshape(-1)


def make_head(wl: Workload, b: int, h: int, perm: Optional[np.ndarray] = None) -> Dict[str, torch.Tensor]:
    """Inputs of one (b, h) slice, block-major, as CPU tensors.

    Returns q, k, v, do ([N, d] bf16) and q_lr, k_lr ([N, r] bf16, integer valued).
    """
    N, d, r = wl.N, wl.d, wl.r
    if perm is None:
        perm = block_major_permutation(wl.latent, wl.block_shape)
    p = torch.from_numpy(perm)
    g = _head_generator(wl, b, h)
    if not wl.planted_locality:
        q = _normal_bf16(g, (N, d))
        k = _normal_bf16(g, (N, d))
        v = _normal_bf16(g, (N, d))
        do = _normal_bf16(g, (N, d))
        q_lr = _int_bf16(g, (N, r), wl.lr_max)
        k_lr = _int_bf16(g, (N, r), wl.lr_max)
        # raster -> block-major
        return {"q": q[p], "k": k[p], "v": v[p], "do": do[p], "q_lr": q_lr[p], "k_lr": k_lr[p]}
    # planted locality: K = K0 + 2 e_n, e shared across each 4x8x8 neighbourhood n
    q = _normal_bf16(g, (N, d))
    k0 = torch.randn((N, d), generator=g, dtype=torch.float32)
    nbh = torch.from_numpy(_neighbourhood_of_token(wl.latent))
    n_nb = int(nbh.max()) + 1
    e = torch.randn((n_nb, d), generator=g, dtype=torch.float32)
    k = (k0 + 2.0 * e[nbh]).to(torch.bfloat16)
    v = _normal_bf16(g, (N, d))
    do = _normal_bf16(g, (N, d))
    R = projection_matrix(wl)
    lim = float(wl.lr_max)
    q_lr = torch.clamp(torch.round(0.5 * (q.float() @ R)), -lim, lim).to(torch.bfloat16)
    k_lr = torch.clamp(torch.round(0.5 * (k.float() @ R)), -lim, lim).to(torch.bfloat16)
    return {"q": q[p], "k": k[p], "v": v[p], "do": do[p], "q_lr": q_lr[p], "k_lr": k_lr[p]}


def make_inputs(wl: Workload, heads: Optional[Sequence[int]] = None, b: int = 0) -> Dict[str, torch.Tensor]:
    """Stacked [1, len(heads), N, *] CPU tensors for the given heads of batch element b."""
    if heads is None:
        heads = range(wl.H)
    perm = block_major_permutation(wl.latent, wl.block_shape)
    slices = [make_head(wl, b, h, perm) for h in heads]
    return {key: torch.stack([s[key] for s in slices], 0).unsqueeze(0).contiguous() for key in slices[0]}


def sample_blocks(n_blocks_total: int, count: int, seed: int = 0) -> np.ndarray:
    """Seeded, sorted choice of `count` distinct query blocks (for sampled parity checks)."""
    rng = np.random.default_rng(seed + 31337)
    count = min(count, n_blocks_total)
    return np.sort(rng.choice(n_blocks_total, size=count, replace=False))


# ---------------------------------------------------------------- fused AdaLN inputs
# (B, N, D) of the AdaLN workloads: the short clip's 16,384 tokens at its attention width
# H * d = 12 * 64 = 768, and the same tokens at a wide MMDiT width of 3,072.
ADALN_WORKLOADS = {
    "short": (1, 16384, 768),
    "wide": (1, 16384, 3072),
}


def make_adaln_inputs(B: int, N: int, D: int, seed: int = 0) -> Dict[str, torch.Tensor]:
    """x [B, N, D], scale [B, D], shift [B, D], dy [B, N, D] as bf16 CPU tensors.

    One CPU generator seeded with ``seed + 15485863``; draw order: x's N(0, 1) entries, one
    N(0, 1) offset and one U(0.5, 3) spread per token (x = spread * entry + offset, so rows
    differ in mean and scale as hidden states do), scale ~ 0.5 N(0, 1), shift ~ N(0, 1),
    dy ~ N(0, 1); all rounded to bf16.
    """
    g = torch.Generator().manual_seed(seed + 15485863)
    e = torch.randn(B, N, D, generator=g)
    off = torch.randn(B, N, 1, generator=g)
    spread = 0.5 + 2.5 * torch.rand(B, N, 1, generator=g)
    x = (spread * e + off).to(torch.bfloat16)
    scale = (0.5 * torch.randn(B, D, generator=g)).to(torch.bfloat16)
    shift = torch.randn(B, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    return {"x": x.contiguous(), "scale": scale.contiguous(), "shift": shift.contiguous(), "dy": dy.contiguous()}


def make_inputs_on_device(wl: Workload, device, heads: Optional[Sequence[int]] = None, b: int = 0
                          ) -> Dict[str, torch.Tensor]:
    """The same workload drawn directly in device memory, for timing runs whose inputs would take
    minutes to draw on the host (the long clip's 24 heads are 6.4 G normal samples).

    Same distributions, draw order, per-(batch, head) seeds, mid-clip planting and block-major
    token order as :func:`make_head`, but the numbers come from torch's device generator
    (Philox), so they differ from the host draw: nothing compares them with the oracle.
    Returns stacked [1, len(heads), N, *] tensors on ``device``.
    """
    if heads is None:
        heads = range(wl.H)
    heads = list(heads)
    N, d, r = wl.N, wl.d, wl.r
    perm = torch.from_numpy(block_major_permutation(wl.latent, wl.block_shape)).to(device)
    names = ("q", "k", "v", "do", "q_lr", "k_lr")
    out = {n: torch.empty((1, len(heads), N, r if n.endswith("_lr") else d), dtype=torch.bfloat16, device=device)
           for n in names}
    R = projection_matrix(wl).to(device) if wl.planted_locality else None
    nbh = torch.from_numpy(_neighbourhood_of_token(wl.latent)).to(device) if wl.planted_locality else None
    for i, h in enumerate(heads):
        g = torch.Generator(device=device)
        g.manual_seed(wl.seed + 7919 * (b * wl.H + h))
        normal = lambda shape: torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if not wl.planted_locality:
            x = {"q": normal((N, d)).to(torch.bfloat16), "k": normal((N, d)).to(torch.bfloat16),
                 "v": normal((N, d)).to(torch.bfloat16), "do": normal((N, d)).to(torch.bfloat16)}
            for n in ("q_lr", "k_lr"):
                x[n] = torch.randint(-wl.lr_max, wl.lr_max + 1, (N, r), generator=g, device=device,
                                     dtype=torch.int32).to(torch.bfloat16)
        else:
            q = normal((N, d)).to(torch.bfloat16)
            k0 = normal((N, d))
            e = normal((int(nbh.max()) + 1, d))
            k = (k0 + 2.0 * e[nbh]).to(torch.bfloat16)
            x = {"q": q, "k": k, "v": normal((N, d)).to(torch.bfloat16), "do": normal((N, d)).to(torch.bfloat16)}
            lim = float(wl.lr_max)
            x["q_lr"] = torch.clamp(torch.round(0.5 * (q.float() @ R)), -lim, lim).to(torch.bfloat16)
            x["k_lr"] = torch.clamp(torch.round(0.5 * (k.float() @ R)), -lim, lim).to(torch.bfloat16)
        for n in names:
            torch.index_select(x[n], 0, perm, out=out[n][0, i])
        del x
    return out
