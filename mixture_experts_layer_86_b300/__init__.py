"""Single-GPU top-k gated Mixture-of-Experts FFN layer for NVIDIA B300.

The compute lives in ``libmoe_b300.so`` (hand-written sm_103a CUDA behind the
C ABI of ``include/moe_b300.h``); ``_native`` is its ctypes binding and
``layer`` holds the caller-side allocation helpers.  ``inputs`` draws the
seeded synthetic workloads.  Importing the package does not load the
library; touching ``_native`` or ``layer`` does, and fails if it is missing.
"""
__all__ = ["inputs", "layer", "_native", "build"]
