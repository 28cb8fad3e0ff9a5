"""CPU oracle for the routed-expert MoE layer (plain numpy, float64 where the pages fix nothing).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
import anything here. It shares no code with the CUDA path. Parity unpinned (by printed values):
the pages print no worked example, so the router's sigmoid/bias/normalisation convention and the
round-up scale rule are readings, pinned only by closed forms, invariants and brute force.
"""
from . import formats, moe  # noqa: F401
