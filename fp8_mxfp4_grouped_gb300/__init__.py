"""Grouped-contiguous FP8 E4M3 x MXFP4 E2M1 MoE expert GEMM for GB300 (sm_103a).

The compute path is the C-ABI library ``libhg.so`` (``include/hg.h``), built
from ``csrc/`` by ``build.py``; ``hg`` is its Python binding.
"""
__all__ = ["hg", "build"]
