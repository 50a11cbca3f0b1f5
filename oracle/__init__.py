"""Float64 CPU oracle for the W4A16 routed-MoE block.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this package: only the tests, the smoke
check and the CPU-baseline leg of the benchmark use it. It shares no code with the CUDA library.
"""
from .moe_oracle import *  # noqa: F401,F403
