"""Seeded synthetic inputs for the sparse MoE FFN layer.

This package only draws random tensors of the right shapes; it holds no arithmetic of the
layer itself, so both the CUDA library's tests/benchmarks and the CPU oracle may use it.
"""
from .gen import WORKLOADS, Workload, make_inputs, workload  # noqa: F401
