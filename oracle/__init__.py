"""fp64 CPU oracle for the routed bit-plane MoE layer (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package; the product library never does.
"""
from . import pw_oracle  # noqa: F401
