"""CPU oracles for DSV's dynamic sparse attention and the fused AdaLN operator -- TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and
its ``--impl reference`` arm) may import, call or execute anything here.  The product
path (the CUDA library and its Python binding) never does, and this package never
imports the product.

Pins (what ties each function to something other than itself) live in ``tests/``:
  estimate / top-k : brute force over all subsets on tiny inputs, a hand-worked
                     fixture in tests/golden/, linearity of the block estimate;
  forward          : torch fp64 scaled_dot_product_attention at density 100 % and
                     with a -inf mask outside the selected set;
  backward         : torch fp64 autograd of the masked dense form, central finite
                     differences, closed forms (sum dV = sum dO, sum dK = 0,
                     unselected keys get zero gradient);
  mass-based k     : the exp2 recipe against 2^x, the target by its defining inequality,
                     sufficiency and minimality of every k, closed forms (equal scores,
                     one dominant key), planted mistakes rejected;
  fused AdaLN      : torch fp64 layer_norm + modulation and its autograd, central finite
                     differences, closed forms (constant rows give y = shift, the per-row
                     invariants sum dx = 0 and sum dx * xhat = 0, d_shift = sum dy),
                     planted mistakes rejected.
"""
from .dsv_oracle import (  # noqa: F401
    block_representatives,
    block_scores,
    default_scale,
    estimate_mass_topk,
    estimate_topk,
    exp2_recipe,
    mass_k,
    mass_target,
    mass_weights,
    run_heads,
    sparse_attn_bwd,
    sparse_attn_fwd,
    topk_select,
)
from .adaln_oracle import adaln_bwd, adaln_fwd, row_stats  # noqa: F401,E402
