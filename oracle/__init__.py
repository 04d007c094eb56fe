"""Float64 CPU oracle of the MoE layer -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs import this package.  Parity status of every function is
stated in ``moe_oracle``'s module docstring.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
