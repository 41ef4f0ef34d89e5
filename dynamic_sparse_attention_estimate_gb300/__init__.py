"""GB300-native (sm_103a) dynamic sparse 3D attention for video DiT training (DSV), and
the fused AdaLN (LayerNorm + modulation) operator of the same training step.

The compute path is a C-ABI CUDA library (``libdsv.so``, entry points declared in
``include/dsv.h``); :mod:`.binding` is a thin ctypes layer over it that passes
device pointers, sizes and the current CUDA stream.  Importing this package does not
load the library; the first call does, and fails loudly if it has not been built.
"""
from .binding import (  # noqa: F401
    DSVError,
    dsv_adaln_bwd,
    dsv_adaln_bwd_workspace,
    dsv_adaln_fwd,
    dsv_estimate_mass_k,
    dsv_estimate_topk,
    dsv_estimate_topk_csr,
    dsv_estimate_topk_workspace,
    dsv_sparse_attn_bwd,
    dsv_sparse_attn_bwd_csr,
    dsv_sparse_attn_bwd_prepare,
    dsv_sparse_attn_bwd_prepared,
    dsv_sparse_attn_bwd_workspace,
    dsv_sparse_attn_fwd,
    dsv_sparse_attn_fwd_csr,
    library_path,
    load_library,
)
