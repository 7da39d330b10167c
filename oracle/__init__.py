"""CPU oracle of the MoE-layer forward pass: test infrastructure only.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package; the CUDA library never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
