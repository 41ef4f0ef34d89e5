"""Plain, slow, fp64 CPU oracle of DSV's dynamic sparse attention.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline leg (and its ``--impl reference`` arm) may import this module.  It
shares no code with the CUDA path and imports nothing from the package.

What it computes follows the DSV pages ("DSV: Exploiting Dynamic Sparsity to
Accelerate Large-Scale Video DiT Training", German and Spanish summaries):

* Section 2A (two-stage algorithm with low-rank estimation): per attention head a
  low-rank pair (Q_lr, K_lr) approximates Q K^T, and the critical keys are found
  from that estimate without forming the full attention matrix.
* Section 2B, "Fused MM & Top-K" kernel: the low-rank product and a top-k
  selection together; O(S*k) memory.
* Section 2B, "Query Grouping": 3D-neighbouring tokens share critical keys, so the
  estimate is made once per group of neighbouring queries (a query block).
* Sparse attention itself (custom fused kernels for estimation and sparse
  attention, Spanish summary section 3): softmax attention restricted to the
  selected keys; training needs its backward too.

Readings where the pages are silent:
  1. the block representative is the SUM of the block's Q_lr rows;
  2. keys are ranked by the raw block logit q_hat . K_lr[j] (no scale/softmax);
  3. ties go to the lower key index;
  4. idx rows are stored in ascending key order;
  5. the softmax scale is 1/sqrt(d); there is no causal mask, no forced self key;
  6. every query attends exactly to its block's selected keys.

Every step is written the obvious way with numpy fp64 (a matmul, a stable sort and
exp/log from numpy are the only library primitives); there is no blocking, fusion
or reordering.  Arrays are per head: tokens on axis 0 in block-major order.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np


def _f64(x) -> np.ndarray:
    """Accept numpy arrays or torch tensors (any float dtype) and return fp64 numpy."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------- estimate + top-k

def block_representatives(q_lr, block: int) -> np.ndarray:
    """q_hat[b] = sum of Q_lr over the tokens of query block b  -> [NB, r].

    Query grouping (section 2B): one representative per group of neighbouring
    queries.  With integer-valued factors this sum is exact in fp64.
    """
    q_lr = _f64(q_lr)
    n, r = q_lr.shape
    assert n % block == 0
    return q_lr.reshape(n // block, block, r).sum(axis=1)


def block_scores(q_hat, k_lr) -> np.ndarray:
    """s[b, j] = q_hat[b] . K_lr[j] for every key j -> [NB, N] (low-rank estimate, section 2A)."""
    return _f64(q_hat) @ _f64(k_lr).T


def topk_select(scores, k: int) -> np.ndarray:
    """For each row: order keys by (-score, key index), keep the first k, return them ascending.

    Section 2B's top-k selection, with ties broken towards the lower key index.
    A stable argsort on -score keeps equal scores in ascending key order.
    """
    scores = _f64(scores)
    order = np.argsort(-scores, axis=1, kind="stable")
    return np.sort(order[:, :k], axis=1).astype(np.int32)


def estimate_topk(q_lr, k_lr, block: int, k: int, blocks: Optional[Iterable[int]] = None) -> np.ndarray:
    """idx[b, :] for every query block (or only the listed ones, in the given order) -> int32 [nb, k]."""
    q_hat = block_representatives(q_lr, block)
    if blocks is not None:
        q_hat = q_hat[np.asarray(list(blocks), dtype=np.int64)]
    k_lr = _f64(k_lr)
    out = np.empty((q_hat.shape[0], k), dtype=np.int32)
    rows_per_step = max(1, (1 << 24) // max(1, k_lr.shape[0]))  # bound the [rows, N] score slab
    for s in range(0, q_hat.shape[0], rows_per_step):
        out[s:s + rows_per_step] = topk_select(block_scores(q_hat[s:s + rows_per_step], k_lr), k)
    return out


# ---------------------------------------------------------------- sparse attention

# ---------------------------------------------------------------- mass-based adaptive k
# DSV pages, German summary section 2A (stage 2) and Spanish "Fase 2": the low-rank
# predictors estimate the critical KV pairs, those that make up ~90 % of the attention score.
# Readings (the pages give no formula):
#   * a block's estimated attention distribution over keys is softmax_j(tau * s[b, j]), with
#     tau = 1/64 by default: s is the SUM over the block's 64 queries, tau/s the mean logit;
#   * the critical set is the shortest prefix of the keys in (score desc, key index asc)
#     order whose estimated mass reaches the fraction `mass` of the total;
#   * the mass is taken in integer weights so that the decision is exactly reproducible:
#     w_j = floor(2^24 * 2^x_j), x_j = tau_log2 * (s_j - max_j s_j) in fp32 (tau_log2 =
#     tau * log2(e) rounded to fp32), 2^x from the fp32 recipe exp2_recipe(); the target is
#     ceil(W * mass_num / 2^16) with W = sum_j w_j and mass_num = round(mass * 2^16).

EXP2_TAYLOR = [np.float32(math.log(2.0) ** i / math.factorial(i)) for i in range(7)]


def exp2_recipe(x) -> np.ndarray:
    """2^x for fp32 x <= 0 by the fixed fp32 recipe both the oracle and the kernels follow:
    n = floor(x), f = x - n (exact), 2^f from its Taylor series to degree 6 in Horner form
    (every product and sum rounded to fp32, nothing fused), then scaled by 2^n (exact)."""
    x = np.asarray(x, dtype=np.float32)
    n = np.floor(x).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(EXP2_TAYLOR[6]) * np.ones_like(f)
    for c in EXP2_TAYLOR[5::-1]:
        p = (p * f).astype(np.float32)
        p = (p + c).astype(np.float32)
    return np.ldexp(p, n.astype(np.int32)).astype(np.float32)


def mass_weights(scores_row, tau_log2: float) -> np.ndarray:
    """Integer weights w_j (uint64) of one block's keys; 0 once 2^x < 2^-30."""
    s = np.asarray(scores_row, dtype=np.float64)
    smax = s.max()
    x = (np.float32(tau_log2) * (s - smax).astype(np.float32)).astype(np.float32)
    w = np.zeros(s.shape, dtype=np.uint64)
    live = x >= np.float32(-30.0)
    w[live] = np.floor(exp2_recipe(x[live]).astype(np.float64) * 2.0 ** 24).astype(np.uint64)
    return w


def mass_target(total: int, mass_num: int) -> int:
    """The smallest integer weight t with t >= total * mass_num / 2^16."""
    return (int(total) * int(mass_num) + 65535) >> 16


def mass_k(scores, tau_log2: float, mass_num: int, dense_num: int = 0) -> np.ndarray:
    """Per block the size of the shortest (score desc, key asc) prefix whose weight reaches
    ceil(W * mass_num / 2^16) -> int32 [NB].

    Per-block sparse/dense switch (the pages decide per block from its sparsity level whether
    sparse attention is used): with dense_num > 0, a block whose k exceeds the fraction
    dense_num / 2^16 of the keys (k * 2^16 > dense_num * N) attends to all N keys."""
    scores = np.asarray(scores, dtype=np.float64)
    out = np.empty(scores.shape[0], dtype=np.int32)
    for b in range(scores.shape[0]):
        order = np.lexsort((np.arange(scores.shape[1]), -scores[b]))
        w = mass_weights(scores[b], tau_log2)[order]
        target = mass_target(int(w.sum()), mass_num)
        cum = np.cumsum(w.astype(object))           # exact integers
        out[b] = int(np.argmax(cum >= target)) + 1
        if dense_num and out[b] * 65536 > dense_num * scores.shape[1]:
            out[b] = scores.shape[1]
    return out


def estimate_mass_topk(q_lr, k_lr, block: int, tau_log2: float, mass_num: int, dense_num: int = 0):
    """Adaptive selection: per block its mass-based k, then its top-k keys (ascending).
    Returns (k per block int32 [NB], list of per-block index arrays)."""
    s = block_scores(block_representatives(q_lr, block), k_lr)
    ks = mass_k(s, tau_log2, mass_num, dense_num)
    return ks, [topk_select(s[b:b + 1], int(ks[b]))[0] for b in range(s.shape[0])]


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def sparse_attn_fwd(q, k, v, idx, block: int, scale: Optional[float] = None,
                    blocks: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of each query over its block's selected keys only.

    For query i in block b:  l_ij = scale * Q_i . K_j  (j in idx[b]),
    LSE_i = m_i + ln sum_j exp(l_ij - m_i) with m_i = max_j l_ij,
    P_ij = exp(l_ij - LSE_i),  O_i = sum_j P_ij V_j.
    Returns O [N, d] and LSE [N] (fp64); rows of blocks not computed are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    idx = idx if isinstance(idx, (list, tuple)) else np.asarray(idx)  # per-block lists may be ragged
    n, d = q.shape
    if scale is None:
        scale = default_scale(d)
    nb = n // block
    blocks = range(nb) if blocks is None else blocks
    o = np.full((n, d), np.nan)
    lse = np.full((n,), np.nan)
    for b in blocks:
        rows = slice(b * block, (b + 1) * block)
        sel = idx[b].astype(np.int64)
        logits = scale * (q[rows] @ k[sel].T)            # [block, k]
        m = logits.max(axis=1, keepdims=True)
        lse_b = m[:, 0] + np.log(np.exp(logits - m).sum(axis=1))
        p = np.exp(logits - lse_b[:, None])
        o[rows] = p @ v[sel]
        lse[rows] = lse_b
    return o, lse


def sparse_attn_bwd(do, q, k, v, idx, block: int, scale: Optional[float] = None,
                    blocks: Optional[Iterable[int]] = None, o=None, lse=None):
    """Gradients of sum(dO * O) w.r.t. Q, K, V for the sparse attention above.

    D_i = dO_i . O_i;  dP_ij = dO_i . V_j;  dS_ij = P_ij (dP_ij - D_i);
    dQ_i = scale sum_j dS_ij K_j;  dK_j = scale sum_i dS_ij Q_i;  dV_j = sum_i P_ij dO_i,
    the last two summed over every query whose block selected key j (0 if none).
    With ``blocks`` given, only those query blocks contribute (the others are taken
    to have dO = 0, which is what zeroing dO outside them does exactly).
    """
    do, q, k, v = _f64(do), _f64(q), _f64(k), _f64(v)
    idx = idx if isinstance(idx, (list, tuple)) else np.asarray(idx)  # per-block lists may be ragged
    n, d = q.shape
    if scale is None:
        scale = default_scale(d)
    nb = n // block
    blocks = list(range(nb)) if blocks is None else list(blocks)
    if o is None or lse is None:
        o, lse = sparse_attn_fwd(q, k, v, idx, block, scale, blocks)
    o, lse = _f64(o), _f64(lse)
    dq = np.zeros((n, d))
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    for b in blocks:
        rows = slice(b * block, (b + 1) * block)
        sel = idx[b].astype(np.int64)
        logits = scale * (q[rows] @ k[sel].T)
        p = np.exp(logits - lse[rows][:, None])
        big_d = (do[rows] * o[rows]).sum(axis=1)
        dp = do[rows] @ v[sel].T
        ds = p * (dp - big_d[:, None])
        dq[rows] = scale * (ds @ k[sel])
        dk[sel] += scale * (ds.T @ q[rows])   # keys in one idx row are distinct
        dv[sel] += p.T @ do[rows]
    return dq, dk, dv


# ---------------------------------------------------------------- whole [B, H, N, *] tensors

def run_heads(fn, *tensors, **kw):
    """Apply a per-head oracle function to every (b, h) slice of [B, H, ...] inputs."""
    first = tensors[0]
    B, H = first.shape[0], first.shape[1]
    outs = []
    for b in range(B):
        row = []
        for h in range(H):
            row.append(fn(*[t[b, h] for t in tensors], **kw))
        outs.append(row)
    return outs
