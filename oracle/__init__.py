"""CPU oracle for the routed top-k MoE experts forward.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg; never by the product path.  It shares no code
with the CUDA library.  See moe_oracle.py for the definitions and the
passages they follow.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import scale_values  # noqa: F401
