"""C-ABI library: builds, loads, exports every symbol include/dsv.h declares, and rejects
invalid calls on the host before launching anything (CPU only: no compute call)."""
import ctypes
import os
import re

import pytest

import dynamic_sparse_attention_estimate_gb300 as pkg
from dynamic_sparse_attention_estimate_gb300.binding import EXPORTED, make_dims

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(REPO, "include", "dsv.h")


@pytest.fixture(scope="module")
def lib():
    from dynamic_sparse_attention_estimate_gb300.build import build
    build()
    return pkg.load_library()


@pytest.fixture
def no_gpu():
    """The validation tests hand the library made-up device addresses (0x1000 and the like),
    which host validation must reject before anything is launched.  That is only safe where no
    GPU could run a launch if validation ever let one through, so they run on GPU-less hosts
    only; the GPU tests cover the same calls with real buffers."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("made-up device addresses are only passed where no GPU is visible")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.dsv_status_string(0) == b"DSV_OK"
    assert lib.dsv_status_string(5) == b"DSV_ERR_DEVICE_CHECK"


def _call_fwd(lib, dims, ptr=0x1000):
    p = ctypes.c_void_p(ptr)
    return lib.dsv_sparse_attn_fwd(ctypes.byref(dims), p, p, p, p, p, p, None, 0, None)


@pytest.mark.parametrize("field,value,status", [
    ("block", 32, 2), ("N", 1000, 1), ("k", 0, 1), ("k", 1025, 1), ("d", 96, 2), ("B", 0, 1),
])
def test_invalid_dims_rejected_before_launch(lib, no_gpu, field, value, status):
    dims = make_dims(1, 2, 1024, 64, 16, 128)
    setattr(dims, field, value)
    assert _call_fwd(lib, dims) == status
    assert lib.dsv_last_error_message()


def test_null_and_misaligned_pointers_rejected(lib, no_gpu):
    dims = make_dims(1, 2, 1024, 64, 16, 128)
    assert lib.dsv_sparse_attn_fwd(ctypes.byref(dims), None, None, None, None, None, None, None, 0, None) == 1
    assert b"NULL" in lib.dsv_last_error_message()
    assert _call_fwd(lib, dims, 0x1004) == 1
    assert b"aligned" in lib.dsv_last_error_message()
    p = ctypes.c_void_p(0x1000)
    bad_r = make_dims(1, 2, 1024, 64, 24, 128)
    assert lib.dsv_estimate_topk(ctypes.byref(bad_r), p, p, p, None, 0, None) == 2


def test_backward_workspace_checks(lib, no_gpu):
    dims = make_dims(1, 12, 16384, 64, 16, 1638)
    rec = lib.dsv_sparse_attn_bwd_workspace(ctypes.byref(dims))
    mn = lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(dims))
    assert 0 < mn < rec
    # partial rows: 12 heads x 256 blocks x 1638 keys x 2 x 64 bf16
    assert rec >= 12 * 256 * 1638 * 2 * 64 * 2
    p = ctypes.c_void_p(0x1000)
    args = [ctypes.byref(dims)] + [p] * 10
    assert lib.dsv_sparse_attn_bwd(*args, None, 0, None) == 3            # no workspace
    assert lib.dsv_sparse_attn_bwd(*args, ctypes.c_void_p(0x1000), mn - 256, None) == 3   # too small
    assert lib.dsv_sparse_attn_bwd(*args, ctypes.c_void_p(0x1010), rec, None) == 3        # misaligned


def test_estimate_needs_no_workspace(lib):
    dims = make_dims(1, 2, 1024, 64, 16, 128)
    assert lib.dsv_estimate_topk_workspace(ctypes.byref(dims)) == 0


def test_mass_selection_arguments_rejected_before_launch(lib, no_gpu):
    dims = make_dims(1, 2, 1024, 64, 16, 1024)
    p = ctypes.c_void_p(0x1000)
    assert lib.dsv_estimate_mass_k(ctypes.byref(dims), p, p, 0.0, 58982, 0, p, p, None, None) == 1       # tau_log2 <= 0
    assert b"tau_log2" in lib.dsv_last_error_message()
    assert lib.dsv_estimate_mass_k(ctypes.byref(dims), p, p, 0.02, 0, 0, p, p, None, None) == 1       # mass_num 0
    assert lib.dsv_estimate_mass_k(ctypes.byref(dims), p, p, 0.02, 65537, 0, p, p, None, None) == 1   # above 1
    assert lib.dsv_estimate_mass_k(ctypes.byref(dims), p, p, 0.02, 58982, 65537, p, p, None, None) == 1  # dense_num
    assert lib.dsv_estimate_mass_k(ctypes.byref(dims), p, p, 0.02, 58982, 0, None, p, None, None) == 1  # no k_row
    assert lib.dsv_estimate_topk_csr(ctypes.byref(dims), p, p, p, None, p, None) == 1           # no rowptr
    bad_r = make_dims(1, 2, 1024, 64, 24, 1024)
    assert lib.dsv_estimate_mass_k(ctypes.byref(bad_r), p, p, 0.02, 58982, 0, p, p, None, None) == 2


def test_adaln_arguments_rejected_before_launch(lib, no_gpu):
    from dynamic_sparse_attention_estimate_gb300.binding import AdalnDims
    p = ctypes.c_void_p(0x1000)
    good = AdalnDims(1, 16, 768, 1e-6)
    for bad, what in ((AdalnDims(1, 16, 12, 1e-6), b"D"), (AdalnDims(1, 16, 8200, 1e-6), b"D"),
                      (AdalnDims(0, 16, 64, 1e-6), b"B and N"), (AdalnDims(1, 0, 64, 1e-6), b"B and N"),
                      (AdalnDims(1, 16, 64, -1.0), b"eps"), (AdalnDims(1, 16, 64, float("nan")), b"eps")):
        assert lib.dsv_adaln_fwd(ctypes.byref(bad), p, p, p, p, None) == 1
        assert what in lib.dsv_last_error_message()
        assert lib.dsv_adaln_bwd_workspace(ctypes.byref(bad)) == 0
    assert lib.dsv_adaln_fwd(ctypes.byref(good), p, None, p, p, None) == 1
    assert b"NULL" in lib.dsv_last_error_message()
    assert lib.dsv_adaln_fwd(ctypes.byref(good), p, p, ctypes.c_void_p(0x1008), p, None) == 1
    assert b"aligned" in lib.dsv_last_error_message()
    need = lib.dsv_adaln_bwd_workspace(ctypes.byref(good))
    assert need >= 2 * 768 * 4      # at least one tile's partial row of d_scale and d_shift
    args = [ctypes.byref(good), p, p, p, p, p, p]
    assert lib.dsv_adaln_bwd(*args, None, 0, None) == 3
    assert lib.dsv_adaln_bwd(*args, p, need - 256, None) == 3
    assert lib.dsv_adaln_bwd(*args, ctypes.c_void_p(0x1010), need, None) == 3


def test_split_backward_needs_a_single_wave_workspace(lib, no_gpu):
    dims = make_dims(1, 12, 16384, 64, 16, 1638)
    p = ctypes.c_void_p(0x1000)
    mn = lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(dims))
    assert lib.dsv_sparse_attn_bwd_prepare(ctypes.byref(dims), p, p, mn, None) == 3      # several waves
    assert b"one wave" in lib.dsv_last_error_message()
    assert lib.dsv_sparse_attn_bwd_prepare(ctypes.byref(dims), None, p, mn, None) == 1   # no idx
    args = [ctypes.byref(dims)] + [p] * 10
    assert lib.dsv_sparse_attn_bwd_prepared(*args, p, mn, None) == 3


def test_noalloc_rejects_a_problem_larger_than_its_scratch(lib, no_gpu):
    """The no-allocation backward holds DSV_NOALLOC_SCRATCH_BYTES (32 MiB) of scratch.  The
    long clip (N = 520,192, d = 128, k = 52,019) needs far more even one query block at a time:
    52,019 bf16 partial rows of 4 d bytes (26.6 MB) plus a fp32 accumulator of 8 d N bytes
    (533 MB) that chains a head's waves.  The call is rejected on the host, before any device
    work, with the reason in the error message."""
    dims = make_dims(1, 4, 520192, 128, 16, 52019)
    need = lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(dims))
    assert need > 8 * 128 * 520192 + 52019 * 4 * 128
    p = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    assert lib.dsv_sparse_attn_bwd_noalloc(ctypes.byref(dims), p, p, p, p, p, p, p, p, p, p, None) == 3
    assert b"no-allocation" in lib.dsv_last_error_message()


def test_noalloc_accepts_what_fits_its_scratch(lib):
    """The shapes the no-allocation backward accepts: a smallest workspace of at most 32 MiB.
    At d = 128 with the largest sparse k (N - 1) that holds up to about N = 21,000 tokens per head.
    With k = N (every key selected) the dense backward needs only D per row (4 N bytes a head)."""
    limit = 32 << 20
    fits = make_dims(1, 1, 20480, 128, 16, 20479)
    too_big = make_dims(1, 1, 22528, 128, 16, 22527)
    assert lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(fits)) <= limit
    assert lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(too_big)) > limit
    dense = make_dims(1, 1, 22528, 128, 16, 22528)
    assert lib.dsv_sparse_attn_bwd_workspace_min(ctypes.byref(dense)) == 4 * 22528
