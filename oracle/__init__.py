"""fp64 CPU oracle for the MoE layer forward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import this
package.  It shares no code with the CUDA path.
"""
from . import moe_oracle  # noqa: F401
