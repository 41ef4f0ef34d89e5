"""The oracle's pins must catch plausible mistakes (CPU only).

Each case takes the oracle's source, plants one mistake by text substitution,
loads the result as a separate module and checks that an independent pin rejects
it.  The real oracle module is never modified.
"""
import importlib.util
import json
import math
import os
import sys
import types

import numpy as np
import pytest
import torch

import oracle.dsv_oracle as real

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SRC = open(real.__file__).read()


def _mutant(old, new):
    assert SRC.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _topk_golden_ok(m):
    g = json.load(open(os.path.join(GOLDEN, "topk_hand.json")))
    q_lr, k_lr = np.array(g["q_lr"], float), np.array(g["k_lr"], float)
    return all(np.array_equal(m.estimate_topk(q_lr, k_lr, g["block"], int(k)), np.array(w)) for k, w in g["idx"].items())


def _masked_case():
    rng = np.random.default_rng(0)
    n, d, block, k = 128, 16, 32, 24
    q, kk, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    idx = np.stack([np.sort(rng.choice(n, size=k, replace=False)) for _ in range(n // block)]).astype(np.int32)
    mask = torch.full((n, n), float("-inf"), dtype=torch.float64)
    for b in range(idx.shape[0]):
        mask[b * block:(b + 1) * block, torch.from_numpy(idx[b].astype(np.int64))] = 0
    return q, kk, v, do, idx, block, mask


def _fwd_ok(m):
    q, kk, v, do, idx, block, mask = _masked_case()
    scale = 1 / math.sqrt(q.shape[1])
    o, _ = m.sparse_attn_fwd(q, kk, v, idx, block, scale)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(kk), t(v), attn_mask=mask, scale=scale)[0, 0]
    return np.allclose(o, ref.numpy(), atol=1e-10)


def _bwd_ok(m):
    q, kk, v, do, idx, block, mask = _masked_case()
    scale = 1 / math.sqrt(q.shape[1])
    grads = m.sparse_attn_bwd(do, q, kk, v, idx, block, scale)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, kk, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                           attn_mask=mask, scale=scale)[0, 0]
    (out * torch.from_numpy(do)).sum().backward()
    return all(np.allclose(a, b.grad.numpy(), atol=1e-9) for a, b in zip(grads, (tq, tk, tv)))


MUTANTS = [
    # (description, old text, new text, pin)
    ("ties to the higher key index", 'order = np.argsort(-scores, axis=1, kind="stable")',
     'order = (scores.shape[1] - 1 - np.argsort(-scores[:, ::-1], axis=1, kind="stable"))', _topk_golden_ok),
    ("representative = first token", "return q_lr.reshape(n // block, block, r).sum(axis=1)",
     "return q_lr.reshape(n // block, block, r)[:, 0, :]", _topk_golden_ok),
    ("smallest instead of largest", 'np.argsort(-scores, axis=1, kind="stable")',
     'np.argsort(scores, axis=1, kind="stable")', _topk_golden_ok),
    ("scale dropped in forward", "logits = scale * (q[rows] @ k[sel].T)            # [block, k]",
     "logits = (q[rows] @ k[sel].T)            # [block, k]", _fwd_ok),
    ("values gathered with query rows", "o[rows] = p @ v[sel]", "o[rows] = p @ v[sel][::-1]", _fwd_ok),
    ("D with wrong sign", "ds = p * (dp - big_d[:, None])", "ds = p * (dp + big_d[:, None])", _bwd_ok),
    ("dK missing scale", "dk[sel] += scale * (ds.T @ q[rows])", "dk[sel] += (ds.T @ q[rows])", _bwd_ok),
    ("dV with dS instead of P", "dv[sel] += p.T @ do[rows]", "dv[sel] += ds.T @ do[rows]", _bwd_ok),
    ("dQ with V instead of K", "dq[rows] = scale * (ds @ k[sel])", "dq[rows] = scale * (ds @ v[sel])", _bwd_ok),
]


def test_real_oracle_passes_every_pin():
    assert _topk_golden_ok(real) and _fwd_ok(real) and _bwd_ok(real)


@pytest.mark.parametrize("desc,old,new,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_planted_mistake(desc, old, new, pin):
    assert not pin(_mutant(old, new)), desc
