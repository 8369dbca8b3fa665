"""The CPU oracle: test infrastructure only (see tffn_oracle.c).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline and
reference legs may import this package.
"""
from .oracle import (ACT_GELU_TANH, ACT_NONE, ACT_RELU, ACT_SILU, act, bf16_to_f64,  # noqa: F401
                     f64_to_bf16, ffn, glu_ffn, lib, moe_ffn, moe_glu_ffn, moe_permute, moe_route)
