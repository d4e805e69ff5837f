"""CPU oracle for the sparse MoE FFN layer (test infrastructure; see moe_oracle.py)."""
from . import moe_oracle  # noqa: F401
