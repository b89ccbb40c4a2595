"""GB300-native (sm_103a) weight-streaming quantised linear layers.

W8 (per-tensor int8 weights, fp32 activations) and T158 (ternary weights
packed five per byte in base 3, int8 absmax activations, exact int32
accumulation) GEMV/GEMM kernels, and a fused Gemma-3-1B-shaped ternary decode
step.  The C ABI is ``include/qlin.h``; ``qlin`` is its Python binding and
``build`` compiles the library.
"""
from . import build, qlin  # noqa: F401

__all__ = ["qlin", "build"]
