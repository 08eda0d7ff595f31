"""GB300-native dense multiply-accumulate D = A*B + C.

FP16/BF16 inputs accumulate in FP32, INT8 in INT32, FP64 in FP64, plus a
batched small-tile form in which one A block is broadcast across a group of
neighbouring batch entries.  The arithmetic runs in hand-written sm_103a CUDA
kernels behind a C ABI (``include/mma_gb300.h``); this package is the thin
Python binding over it (argument marshalling only) plus the seeded input
generator.  The CUDA library is loaded on first use; if it is missing, every
compute call raises -- there is no CPU fallback.
"""
from .binding import (gemm, gemm_ex, gemm_batched, gemm_i8_ex, library_path, load,  # noqa: F401
                      MMAError)

__all__ = ["gemm", "gemm_ex", "gemm_batched", "gemm_i8_ex", "load", "library_path", "MMAError"]
