"""Sparse Mixture-of-Experts FFN layer, forward pass, for one NVIDIA B300 (sm_103a).

The compute lives in ``libmoe.so`` (hand-written CUDA; C ABI in ``include/moe.h``); ``moe``
is its ctypes binding.  Importing this package does not load the library; the first call does.
"""
from . import moe  # noqa: F401
