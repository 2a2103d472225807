"""Float64 CPU oracle of the DeepSeekMoE layer forward (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import
this package; the CUDA library never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
