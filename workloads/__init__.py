"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package draws inputs only (hidden states, router output, expert outputs).
It holds none of the dispatch/combine arithmetic.
"""
from .gen import CONFIGS, Workload, make_workload, random_case, expert_output, bf16_bits_to_f32

__all__ = ["CONFIGS", "Workload", "make_workload", "random_case", "expert_output", "bf16_bits_to_f32"]
