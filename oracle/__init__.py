"""CPU oracle of the MoE SwiGLU FFN forward (test infrastructure only).

Only tests/, the smoke check in __graft_entry__ and bench.py's cpu_baseline /
reference leg may import this package; the product path never does.
"""
from . import moe_oracle  # noqa: F401
