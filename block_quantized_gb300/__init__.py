"""block_quantized_gb300 -- GGML-style block-quantized GEMV/GEMM for GB300.

The compute path is the CUDA library libgq.so (include/gq.h); ``gq`` is its
Python binding and ``inputs`` holds the seeded synthetic input generators.
"""
from . import gq  # noqa: F401  (binding only; the library loads on first call)

__all__ = ["gq"]
