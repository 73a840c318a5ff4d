"""CPU oracle for the sparse-MoE layer forward (test infrastructure; see moe_oracle.py)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import PLAIN, BIAS_SELECT, GUMBEL, TIE_MARGIN  # noqa: F401
