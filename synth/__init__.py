"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This package holds no arithmetic of the method (no decode, no GEMM, no plan):
it draws routing ids and values and quantises them into the operand codes
that both the CUDA path and the CPU oracle consume.
"""
from .inputs import (CONFIGS, Case, make_case, make_routing, make_weights,
                     make_acts, quantize_acts, quantize_weights)

__all__ = ["CONFIGS", "Case", "make_case", "make_routing", "make_weights",
           "make_acts", "quantize_acts", "quantize_weights"]
