"""fp64 CPU oracle of the routed-MoE forward layer (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg and
reference arm may import this package. It shares no code with the CUDA
library and imports nothing from it.

Parity status of each function against what the pages and the mathematics fix
is recorded in tests/test_oracle_pins.py (every function here is pinned there).
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
