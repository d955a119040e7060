"""fp64 CPU oracle of the MoE-LoRA layer -- test infrastructure only (see oracle.py)."""
from .oracle import Oracle, build, load  # noqa: F401
