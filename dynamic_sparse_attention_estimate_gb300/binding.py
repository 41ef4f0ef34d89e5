"""ctypes binding of libdsv.so (the C ABI declared in include/dsv.h).

Argument marshalling only: each function checks dtypes/shapes of the torch tensors it
is given, allocates outputs with torch on the input's device, and passes raw device
pointers, sizes and the current CUDA stream to the library.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libdsv.so"
_lib = None

DSV_OK = 0
STATUS_NAMES = {0: "DSV_OK", 1: "DSV_ERR_INVALID_ARG", 2: "DSV_ERR_UNSUPPORTED", 3: "DSV_ERR_WORKSPACE",
                4: "DSV_ERR_CUDA", 5: "DSV_ERR_DEVICE_CHECK"}

EXPORTED = (
    "dsv_estimate_topk_workspace", "dsv_estimate_topk", "dsv_sparse_attn_fwd",
    "dsv_sparse_attn_bwd_workspace", "dsv_sparse_attn_bwd_workspace_min", "dsv_sparse_attn_bwd",
    "dsv_status_string", "dsv_last_error_message", "dsv_last_device_status",
    "dsv_profile_enable", "dsv_profile_read", "dsv_sparse_attn_bwd_noalloc",
    "dsv_estimate_mass_k", "dsv_estimate_topk_csr", "dsv_sparse_attn_fwd_csr",
    "dsv_sparse_attn_bwd_csr_workspace", "dsv_sparse_attn_bwd_csr", "dsv_csr_launch_order",
    "dsv_adaln_fwd", "dsv_adaln_bwd_workspace", "dsv_adaln_bwd",
    "dsv_sparse_attn_bwd_prepare", "dsv_sparse_attn_bwd_prepared", "dsv_sparse_attn_fwd_workspace",
)


class DSVError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" + (f" ({detail})" if detail else ""))


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64),
                ("d", ctypes.c_int64), ("r", ctypes.c_int64), ("block", ctypes.c_int64),
                ("k", ctypes.c_int64), ("scale", ctypes.c_float)]


class AdalnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("N", ctypes.c_int64), ("D", ctypes.c_int64), ("eps", ctypes.c_float)]


def library_path() -> str:
    """The in-tree libdsv.so, or the file the DSV_LIBRARY variable names (another build of the same
    sources, e.g. one made with different compiler flags)."""
    return os.environ.get("DSV_LIBRARY") or os.path.join(_HERE, _LIB_NAME)


def load_library(path: Optional[str] = None):
    """Load libdsv.so (once).  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} not found: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    dp = ctypes.POINTER(Dims)
    lib.dsv_estimate_topk_workspace.argtypes = [dp]
    lib.dsv_estimate_topk_workspace.restype = sz
    lib.dsv_estimate_topk.argtypes = [dp, vp, vp, vp, vp, sz, vp]
    lib.dsv_estimate_topk.restype = st
    lib.dsv_sparse_attn_fwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dsv_sparse_attn_fwd.restype = st
    lib.dsv_sparse_attn_fwd_workspace.argtypes = [dp]
    lib.dsv_sparse_attn_fwd_workspace.restype = sz
    lib.dsv_sparse_attn_bwd_workspace.argtypes = [dp]
    lib.dsv_sparse_attn_bwd_workspace.restype = sz
    lib.dsv_sparse_attn_bwd_workspace_min.argtypes = [dp]
    lib.dsv_sparse_attn_bwd_workspace_min.restype = sz
    lib.dsv_sparse_attn_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dsv_sparse_attn_bwd.restype = st
    lib.dsv_status_string.argtypes = [st]
    lib.dsv_status_string.restype = ctypes.c_char_p
    lib.dsv_last_error_message.argtypes = []
    lib.dsv_last_error_message.restype = ctypes.c_char_p
    lib.dsv_last_device_status.argtypes = [vp]
    lib.dsv_last_device_status.restype = st
    lib.dsv_sparse_attn_bwd_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.dsv_sparse_attn_bwd_noalloc.restype = st
    lib.dsv_estimate_mass_k.argtypes = [dp, vp, vp, ctypes.c_float, ctypes.c_uint32, ctypes.c_uint32, vp, vp, vp, vp]
    lib.dsv_estimate_mass_k.restype = st
    lib.dsv_estimate_topk_csr.argtypes = [dp, vp, vp, vp, vp, vp, vp]
    lib.dsv_estimate_topk_csr.restype = st
    lib.dsv_csr_launch_order.argtypes = [dp, vp, vp, vp]
    lib.dsv_csr_launch_order.restype = st
    lib.dsv_sparse_attn_fwd_csr.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.dsv_sparse_attn_fwd_csr.restype = st
    lib.dsv_sparse_attn_bwd_csr_workspace.argtypes = [dp, ctypes.c_int64]
    lib.dsv_sparse_attn_bwd_csr_workspace.restype = sz
    lib.dsv_sparse_attn_bwd_csr.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, vp, sz,
                                            vp]
    lib.dsv_sparse_attn_bwd_csr.restype = st
    lib.dsv_sparse_attn_bwd_prepare.argtypes = [dp, vp, vp, sz, vp]
    lib.dsv_sparse_attn_bwd_prepare.restype = st
    lib.dsv_sparse_attn_bwd_prepared.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dsv_sparse_attn_bwd_prepared.restype = st
    ap = ctypes.POINTER(AdalnDims)
    lib.dsv_adaln_fwd.argtypes = [ap, vp, vp, vp, vp, vp]
    lib.dsv_adaln_fwd.restype = st
    lib.dsv_adaln_bwd_workspace.argtypes = [ap]
    lib.dsv_adaln_bwd_workspace.restype = sz
    lib.dsv_adaln_bwd.argtypes = [ap, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dsv_adaln_bwd.restype = st
    lib.dsv_profile_enable.argtypes = [st]
    lib.dsv_profile_enable.restype = st
    lib.dsv_profile_read.argtypes = [ctypes.c_char_p, sz]
    lib.dsv_profile_read.restype = sz
    if path is None:
        _lib = lib
    return lib


def make_dims(B, H, N, d, r, k, block=64, scale: Optional[float] = None) -> Dims:
    return Dims(int(B), int(H), int(N), int(d), int(r), int(block), int(k),
                float(scale) if scale is not None else 0.0)


def _check(status: int, what: str):
    if status != DSV_OK:
        lib = load_library()
        msg = lib.dsv_last_error_message()
        raise DSVError(status, what, msg.decode() if msg else "")


def _stream_ptr(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: need a contiguous CUDA {dtype} tensor with {ndim} dims, got "
                         f"{t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()} device={t.device}")


# ---------------------------------------------------------------- entry points (same names as the C ABI)

def dsv_estimate_topk_workspace(dims: Dims) -> int:
    return int(load_library().dsv_estimate_topk_workspace(ctypes.byref(dims)))


def dsv_estimate_topk(q_lr: torch.Tensor, k_lr: torch.Tensor, k: int, block: int = 64,
                      idx: Optional[torch.Tensor] = None) -> torch.Tensor:
    """idx [B, H, N/block, k] int32 of the top-k keys per query block (ascending)."""
    _need(q_lr, "q_lr", torch.bfloat16, 4)
    _need(k_lr, "k_lr", torch.bfloat16, 4)
    B, H, N, r = q_lr.shape
    if k_lr.shape != q_lr.shape:
        raise ValueError("q_lr and k_lr must have the same shape")
    dims = make_dims(B, H, N, 0, r, k, block)
    if idx is None:
        idx = torch.empty((B, H, max(N // block, 0), int(k)), dtype=torch.int32, device=q_lr.device)
    lib = load_library()
    ws_bytes = int(lib.dsv_estimate_topk_workspace(ctypes.byref(dims)))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q_lr.device) if ws_bytes else None
    _check(lib.dsv_estimate_topk(ctypes.byref(dims), _ptr(q_lr), _ptr(k_lr), _ptr(idx), _ptr(ws), ws_bytes,
                                 _stream_ptr(q_lr)), "dsv_estimate_topk")
    return idx


def mass_parameters(tau: float, mass: float) -> Tuple[float, int]:
    """(tau_log2, mass_num) as dsv_estimate_mass_k takes them: tau * log2(e) rounded to fp32,
    and the mass fraction in units of 2^-16 (rounded, 1 .. 65536)."""
    import numpy as np
    tau_log2 = float(np.float32(float(tau) / 0.6931471805599453))
    mass_num = int(min(65536, max(1, round(float(mass) * 65536))))
    return tau_log2, mass_num


def dsv_estimate_mass_k(q_lr: torch.Tensor, k_lr: torch.Tensor, tau: float = 1.0 / 64, mass: float = 0.9,
                        block: int = 64, out: Optional[Tuple] = None, with_order: bool = True,
                        dense_above: Optional[float] = None):
    """(k_row int32 [B, H, N/block], rowptr int64 [B*H*N/block + 1], order int32 [B*H*N/block] or
    None): per query block the smallest number of top keys that carry the fraction `mass` of
    the estimated attention mass softmax_j(tau s[b, j]), the CSR offsets, and a launch order
    (longest rows first) for the CSR attention calls (see include/dsv.h).  With `dense_above`, a block whose k exceeds
    that fraction of the keys attends to all of them (the per-block sparse/dense switch)."""
    _need(q_lr, "q_lr", torch.bfloat16, 4)
    _need(k_lr, "k_lr", torch.bfloat16, 4)
    B, H, N, r = q_lr.shape
    if k_lr.shape != q_lr.shape:
        raise ValueError("q_lr and k_lr must have the same shape")
    dims = make_dims(B, H, N, 0, r, max(N, 1), block)
    NB = max(N // block, 0)
    if out is None:
        k_row = torch.empty((B, H, NB), dtype=torch.int32, device=q_lr.device)
        rowptr = torch.empty((B * H * NB + 1,), dtype=torch.int64, device=q_lr.device)
        order = torch.empty((B * H * NB,), dtype=torch.int32, device=q_lr.device) if with_order else None
    else:
        k_row, rowptr, order = out
    tau_log2, mass_num = mass_parameters(tau, mass)
    dense_num = 0 if dense_above is None else int(min(65536, max(0, round(float(dense_above) * 65536))))
    _check(load_library().dsv_estimate_mass_k(ctypes.byref(dims), _ptr(q_lr), _ptr(k_lr), tau_log2, mass_num,
                                              dense_num, _ptr(k_row), _ptr(rowptr), _ptr(order), _stream_ptr(q_lr)),
           "dsv_estimate_mass_k")
    return k_row, rowptr, order


def dsv_estimate_topk_csr(q_lr: torch.Tensor, k_lr: torch.Tensor, k_row: torch.Tensor, rowptr: torch.Tensor,
                          block: int = 64, cols: Optional[torch.Tensor] = None) -> torch.Tensor:
    """cols int32 [rowptr[-1]]: row i's k_row[i] top keys (ascending) at cols[rowptr[i]:rowptr[i+1]].
    Without `cols` the total is read from the device (a synchronisation)."""
    _need(q_lr, "q_lr", torch.bfloat16, 4)
    _need(k_lr, "k_lr", torch.bfloat16, 4)
    B, H, N, r = q_lr.shape
    dims = make_dims(B, H, N, 0, r, max(N, 1), block)
    if cols is None:
        cols = torch.empty((int(rowptr[-1].item()),), dtype=torch.int32, device=q_lr.device)
    _check(load_library().dsv_estimate_topk_csr(ctypes.byref(dims), _ptr(q_lr), _ptr(k_lr), _ptr(k_row), _ptr(rowptr),
                                                _ptr(cols), _stream_ptr(q_lr)), "dsv_estimate_topk_csr")
    return cols


def dsv_sparse_attn_fwd_workspace(dims: Dims) -> int:
    return int(load_library().dsv_sparse_attn_fwd_workspace(ctypes.byref(dims)))


def dsv_sparse_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, idx: Optional[torch.Tensor], block: int = 64,
                        scale: Optional[float] = None, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                        workspace: Optional[torch.Tensor] = None):
    """(O bf16 [B,H,N,d], LSE fp32 [B,H,N]) of softmax attention over the selected keys.  Without a
    workspace argument the workspace the library asks for (for key passes) is allocated here."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, H, N, d = q.shape
    if idx is None:   # every key selected (k = N): the dense path, which reads no idx
        kk = N
    else:
        _need(idx, "idx", torch.int32, 4)
        kk = idx.shape[3]
    dims = make_dims(B, H, N, d, 0, kk, block, scale)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    lib = load_library()
    if workspace is None:
        nbytes = int(lib.dsv_sparse_attn_fwd_workspace(ctypes.byref(dims)))
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    _check(lib.dsv_sparse_attn_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse),
                                   _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream_ptr(q)),
           "dsv_sparse_attn_fwd")
    return o, lse


def dsv_sparse_attn_bwd_workspace(dims: Dims, minimum: bool = False) -> int:
    lib = load_library()
    f = lib.dsv_sparse_attn_bwd_workspace_min if minimum else lib.dsv_sparse_attn_bwd_workspace
    return int(f(ctypes.byref(dims)))


def dsv_sparse_attn_bwd(do: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                        lse: torch.Tensor, idx: Optional[torch.Tensor], block: int = 64, scale: Optional[float] = None,
                        workspace: Optional[torch.Tensor] = None, out=None):
    """(dQ, dK, dV) bf16 [B,H,N,d]; dK/dV reduced deterministically per key."""
    for t, n in ((do, "do"), (q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, n, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, H, N, d = q.shape
    if idx is None:   # every key selected (k = N): the dense backward, which reads no idx
        kk = N
    else:
        _need(idx, "idx", torch.int32, 4)
        kk = idx.shape[3]
    dims = make_dims(B, H, N, d, 0, kk, block, scale)
    lib = load_library()
    if workspace is None:
        nbytes = int(lib.dsv_sparse_attn_bwd_workspace(ctypes.byref(dims)))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    _check(lib.dsv_sparse_attn_bwd(ctypes.byref(dims), _ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                   _ptr(idx), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                                   _stream_ptr(q)), "dsv_sparse_attn_bwd")
    return dq, dk, dv


def dsv_sparse_attn_bwd_prepare(idx: torch.Tensor, d: int, workspace: torch.Tensor, block: int = 64) -> None:
    """First half of a split backward: the key-major rank structure of idx, written into `workspace`
    (which must hold every head in one wave: dsv_sparse_attn_bwd_workspace).  Reads idx only, so it
    may run on another stream beside the forward; order dsv_sparse_attn_bwd_prepared after it."""
    _need(idx, "idx", torch.int32, 4)
    B, H, NB, kk = idx.shape
    dims = make_dims(B, H, NB * block, d, 0, kk, block)
    _check(load_library().dsv_sparse_attn_bwd_prepare(ctypes.byref(dims), _ptr(idx), _ptr(workspace),
                                                      workspace.numel(), _stream_ptr(idx)),
           "dsv_sparse_attn_bwd_prepare")


def dsv_sparse_attn_bwd_prepared(do: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                 o: torch.Tensor, lse: torch.Tensor, idx: torch.Tensor, workspace: torch.Tensor,
                                 block: int = 64, scale: Optional[float] = None, out=None):
    """Second half of a split backward, on the workspace dsv_sparse_attn_bwd_prepare filled: the same
    (dQ, dK, dV) as dsv_sparse_attn_bwd, bit for bit."""
    for t, n in ((do, "do"), (q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, n, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    _need(idx, "idx", torch.int32, 4)
    B, H, N, d = q.shape
    dims = make_dims(B, H, N, d, 0, idx.shape[3], block, scale)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    _check(load_library().dsv_sparse_attn_bwd_prepared(ctypes.byref(dims), _ptr(do), _ptr(q), _ptr(k), _ptr(v),
                                                       _ptr(o), _ptr(lse), _ptr(idx), _ptr(dq), _ptr(dk), _ptr(dv),
                                                       _ptr(workspace), workspace.numel(), _stream_ptr(q)),
           "dsv_sparse_attn_bwd_prepared")
    return dq, dk, dv


def dsv_csr_launch_order(rowptr: torch.Tensor, B: int, H: int, N: int, block: int = 64) -> torch.Tensor:
    """int32 [B*H*N/block]: the CSR rows by descending number of 128-key chunks."""
    _need(rowptr, "rowptr", torch.int64, 1)
    dims = make_dims(B, H, N, 0, 16, max(N, 1), block)
    order = torch.empty((B * H * (N // block),), dtype=torch.int32, device=rowptr.device)
    _check(load_library().dsv_csr_launch_order(ctypes.byref(dims), _ptr(rowptr), _ptr(order), _stream_ptr(rowptr)),
           "dsv_csr_launch_order")
    return order


def dsv_sparse_attn_fwd_csr(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rowptr: torch.Tensor, cols: torch.Tensor,
                            block: int = 64, scale: Optional[float] = None,
                            out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None, order: Optional[torch.Tensor] = None):
    """(O, LSE) of attention where query block i attends to cols[rowptr[i]:rowptr[i+1]]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _need(rowptr, "rowptr", torch.int64, 1)
    _need(cols, "cols", torch.int32, 1)
    B, H, N, d = q.shape
    dims = make_dims(B, H, N, d, 0, max(N, 1), block, scale)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    _check(load_library().dsv_sparse_attn_fwd_csr(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(rowptr),
                                                  _ptr(cols), _ptr(order), _ptr(o), _ptr(lse), _stream_ptr(q)),
           "dsv_sparse_attn_fwd_csr")
    return o, lse


def dsv_sparse_attn_bwd_csr_workspace(dims: Dims, total_pairs: int) -> int:
    return int(load_library().dsv_sparse_attn_bwd_csr_workspace(ctypes.byref(dims), int(total_pairs)))


def dsv_sparse_attn_bwd_csr(do: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                            lse: torch.Tensor, rowptr: torch.Tensor, cols: torch.Tensor, block: int = 64,
                            scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None, out=None,
                            order: Optional[torch.Tensor] = None):
    """(dQ, dK, dV) for the CSR attention above (one wave; total pairs = cols.numel())."""
    for t, n in ((do, "do"), (q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, n, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    _need(rowptr, "rowptr", torch.int64, 1)
    _need(cols, "cols", torch.int32, 1)
    B, H, N, d = q.shape
    dims = make_dims(B, H, N, d, 0, max(N, 1), block, scale)
    pairs = cols.numel()
    lib = load_library()
    if workspace is None:
        nbytes = int(lib.dsv_sparse_attn_bwd_csr_workspace(ctypes.byref(dims), pairs))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    _check(lib.dsv_sparse_attn_bwd_csr(ctypes.byref(dims), _ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       _ptr(rowptr), _ptr(cols), _ptr(order), pairs, _ptr(dq), _ptr(dk), _ptr(dv),
                                       _ptr(workspace),
                                       workspace.numel(), _stream_ptr(q)), "dsv_sparse_attn_bwd_csr")
    return dq, dk, dv


# ---------------------------------------------------------------- fused AdaLN

def _adaln_dims(x: torch.Tensor, eps: float) -> AdalnDims:
    B, N, D = x.shape
    return AdalnDims(int(B), int(N), int(D), float(eps))


def _need_mod(t: torch.Tensor, name: str, x: torch.Tensor):
    _need(t, name, torch.bfloat16, 2)
    if t.shape != (x.shape[0], x.shape[2]):
        raise ValueError(f"{name} must be [B, D] = {(x.shape[0], x.shape[2])}, got {tuple(t.shape)}")


def dsv_adaln_fwd(x: torch.Tensor, scale: torch.Tensor, shift: torch.Tensor, eps: float = 1e-6,
                  y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y [B, N, D] bf16 = LayerNorm(x) * (1 + scale[b]) + shift[b] (see include/dsv.h)."""
    _need(x, "x", torch.bfloat16, 3)
    _need_mod(scale, "scale", x)
    _need_mod(shift, "shift", x)
    if y is None:
        y = torch.empty_like(x)
    dims = _adaln_dims(x, eps)
    _check(load_library().dsv_adaln_fwd(ctypes.byref(dims), _ptr(x), _ptr(scale), _ptr(shift), _ptr(y),
                                        _stream_ptr(x)), "dsv_adaln_fwd")
    return y


def dsv_adaln_bwd_workspace(B: int, N: int, D: int, eps: float = 1e-6) -> int:
    dims = AdalnDims(int(B), int(N), int(D), float(eps))
    return int(load_library().dsv_adaln_bwd_workspace(ctypes.byref(dims)))


def dsv_adaln_bwd(x: torch.Tensor, scale: torch.Tensor, dy: torch.Tensor, eps: float = 1e-6,
                  out: Optional[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]] = None,
                  workspace: Optional[torch.Tensor] = None):
    """(dx bf16 [B, N, D], d_scale fp32 [B, D], d_shift fp32 [B, D]) for the loss gradient dy."""
    _need(x, "x", torch.bfloat16, 3)
    _need(dy, "dy", torch.bfloat16, 3)
    _need_mod(scale, "scale", x)
    if dy.shape != x.shape:
        raise ValueError("dy must have the shape of x")
    B, N, D = x.shape
    if out is None:
        out = (torch.empty_like(x), torch.empty((B, D), dtype=torch.float32, device=x.device),
               torch.empty((B, D), dtype=torch.float32, device=x.device))
    dx, d_scale, d_shift = out
    dims = _adaln_dims(x, eps)
    lib = load_library()
    need = int(lib.dsv_adaln_bwd_workspace(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check(lib.dsv_adaln_bwd(ctypes.byref(dims), _ptr(x), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale),
                             _ptr(d_shift), _ptr(workspace), workspace.numel(), _stream_ptr(x)), "dsv_adaln_bwd")
    return dx, d_scale, d_shift


def dsv_last_device_status(device: Optional[torch.device] = None) -> int:
    stream = torch.cuda.current_stream(device).cuda_stream
    return int(load_library().dsv_last_device_status(stream))


def dsv_profile_enable(on: bool = True) -> None:
    _check(load_library().dsv_profile_enable(1 if on else 0), "dsv_profile_enable")


def dsv_profile_read() -> dict:
    """{kernel name: (launches, total device ms)} since the previous read."""
    lib = load_library()
    need = int(lib.dsv_profile_read(None, 0))
    buf = ctypes.create_string_buffer(max(need, 1) + 4096)
    lib.dsv_profile_read(buf, len(buf))
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        out[name] = (int(n), float(ms))
    return out
