"""Shared helpers for the GPU parity tests (compare CUDA outputs with the fp64 oracle)."""
import numpy as np
import pytest
import torch

# Tolerances for bf16 outputs computed with fp32 accumulation vs the fp64 oracle.
MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_MAX_ABS = 1e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from dynamic_sparse_attention_estimate_gb300.build import build
    build()
    return torch.device("cuda:0")


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got, ref):
    got = np64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


# Edge cases (k = 1 and the like) produce outputs far above 1 in magnitude, where the bf16
# spacing alone exceeds the absolute bound; there the bound grows by 2^-7 |ref| per element
# (four bf16 half-ulps: the output rounding plus bf16 operands inside the products).
EDGE_REL_ELEM = 2.0 ** -7


def assert_close(name, got, ref, max_abs=MAX_ABS, rel_l2=REL_L2, rel_elem=0.0):
    m, r = errors(got, ref)
    if rel_elem:
        g = np64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        excess = float((np.abs(g - ref) - (max_abs + rel_elem * np.abs(ref))).max())
        assert excess <= 0 and r <= rel_l2, f"{name}: max-abs {m:.3e} exceeds {max_abs} + {rel_elem} |ref| by {excess:.3e}, rel-L2 {r:.3e}"
        return m, r
    assert m <= max_abs and r <= rel_l2, f"{name}: max-abs {m:.3e} (<= {max_abs}), rel-L2 {r:.3e} (<= {rel_l2})"
    return m, r


def check_idx_invariants(idx, N):
    """Every row: k distinct ascending entries in [0, N) (checked on the device)."""
    assert int(idx.min()) >= 0 and int(idx.max()) < N
    if idx.shape[-1] > 1:
        assert bool((idx[..., 1:] > idx[..., :-1]).all())
