"""CPU oracle for the AWQ W4A16 linear layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.
"""
from .awq_oracle import *  # noqa: F401,F403
from .awq_oracle import (GROUP, W_BIT, QMAX, N_GRID, TOL_REL, MSE_REL,  # noqa: F401
                         absmean, alpha_grid, channel_scales, quantize,
                         pack_codes, unpack_codes, pack_zeros, unpack_zeros,
                         awq_pack, dequant, scaled_activations, linear,
                         ulp_fp16, tolerance, row_errors, search, gram,
                         row_errors_gram, SILU_LIP, silu, silu_mul_linear,
                         fold_inv_scales, CLIP_MIN, clip_ratios, quantize_clipped,
                         group_gram, clip_search)
