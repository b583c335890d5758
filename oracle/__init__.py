"""CPU oracle for the sparse MoE layer forward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may import
this package. It shares no code with the CUDA path and imports nothing from it.
"""
from . import moe_oracle  # noqa: F401
