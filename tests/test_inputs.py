"""Host-side input generation: token layout and seeded draws (CPU only)."""
import numpy as np
import pytest
import torch

from dynamic_sparse_attention_estimate_gb300.inputs import (
    BLOCK, WORKLOADS, block_major_permutation, make_head, make_inputs, sample_blocks)


def _coords(latent, raster_idx):
    T, Hh, W = latent
    return np.stack([raster_idx // (Hh * W), (raster_idx // W) % Hh, raster_idx % W], axis=1)


def test_every_permutation_is_a_bijection():
    for wl in WORKLOADS.values():
        perm = block_major_permutation(wl.latent, wl.block_shape)
        assert perm.size == wl.N
        assert np.array_equal(np.sort(perm), np.arange(wl.N))


def test_cube_blocks_are_4x4x4_neighbourhoods():
    wl = WORKLOADS["short"]
    perm = block_major_permutation(wl.latent, wl.block_shape)
    c = _coords(wl.latent, perm).reshape(wl.NB, BLOCK, 3)
    extent = c.max(axis=1) - c.min(axis=1)
    assert np.all(extent == 3)


def test_long_workload_tail_frames_use_1x8x8_tiles():
    wl = WORKLOADS["long"]
    perm = block_major_permutation(wl.latent, wl.block_shape)
    c = _coords(wl.latent, perm).reshape(wl.NB, BLOCK, 3)
    extent = c.max(axis=1) - c.min(axis=1)
    n_cube_blocks = (124 // 4) * (64 // 4) * (64 // 4)
    assert np.all(extent[:n_cube_blocks] == 3)
    assert np.all(extent[n_cube_blocks:] == np.array([0, 7, 7]))
    assert wl.NB == 8128


def test_tiny_uses_consecutive_raster_blocks():
    wl = WORKLOADS["tiny"]
    assert np.array_equal(block_major_permutation(wl.latent, wl.block_shape), np.arange(wl.N))


def test_draws_are_seeded_shaped_and_integer_factors_in_range():
    wl = WORKLOADS["tiny"]
    a = make_inputs(wl)
    b = make_inputs(wl)
    for key in a:
        assert torch.equal(a[key], b[key])
        assert a[key].dtype == torch.bfloat16
    assert a["q"].shape == (1, 2, 1024, 64) and a["q_lr"].shape == (1, 2, 1024, 16)
    lr = a["q_lr"].float()
    assert torch.equal(lr, lr.round()) and lr.abs().max() <= 4
    # heads are independent streams: generating head 1 alone gives the same slice
    alone = make_head(wl, 0, 1)
    assert torch.equal(alone["k"], a["k"][0, 1])


def test_k_from_density_is_floor():
    wl = WORKLOADS["sweep"]
    assert [wl.with_density(x).k for x in (0.05, 0.10, 0.20, 1.0)] == [6553, 13107, 26214, 131072]
    assert WORKLOADS["short"].k == 1638 and WORKLOADS["long"].k == 52019


def test_sample_blocks_sorted_distinct():
    s = sample_blocks(8128, 64)
    assert s.size == 64 and np.all(np.diff(s) > 0) and s.max() < 8128


def test_adaln_draws_are_seeded_shaped_and_spread_per_token():
    from dynamic_sparse_attention_estimate_gb300.inputs import ADALN_WORKLOADS, make_adaln_inputs
    a, b = make_adaln_inputs(2, 300, 64), make_adaln_inputs(2, 300, 64)
    for n in ("x", "scale", "shift", "dy"):
        assert a[n].dtype == torch.bfloat16 and a[n].is_contiguous()
        assert torch.equal(a[n], b[n])                        # same seed, same draws
    assert a["x"].shape == a["dy"].shape == (2, 300, 64) and a["scale"].shape == a["shift"].shape == (2, 64)
    assert not torch.equal(make_adaln_inputs(2, 300, 64, seed=1)["x"], a["x"])
    # tokens differ in mean and spread (offset N(0,1), spread U(0.5, 3)), as hidden states do
    x = a["x"].float()
    sd = x.std(dim=-1)
    assert float(sd.min()) > 0.3 and float(sd.max()) < 4.0 and float(sd.max() / sd.min()) > 2.0
    assert float(x.mean(dim=-1).std()) > 0.5
    assert set(ADALN_WORKLOADS) == {"short", "wide"}
    assert all(D % 8 == 0 for (_, _, D) in ADALN_WORKLOADS.values())


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_device_draw_follows_the_host_recipe(name):
    """make_inputs_on_device runs the host recipe step for step: given the host's generator it
    reproduces make_inputs exactly (on a GPU only the generator's numbers differ)."""
    from dynamic_sparse_attention_estimate_gb300.inputs import make_inputs_on_device
    wl = WORKLOADS[name]
    heads = [0, 1] if name == "tiny" else [3]
    a = make_inputs(wl, heads=heads)
    b = make_inputs_on_device(wl, torch.device("cpu"), heads=heads)
    for key in a:
        assert torch.equal(a[key], b[key]), key
