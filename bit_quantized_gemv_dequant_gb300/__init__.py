"""Quantized GEMV with fused dequantization for GB300 (sm_103a).

The compute lives in the CUDA library libqgemv.so (C ABI in include/qgemv.h);
this package is a thin ctypes binding over it. The library is loaded on first
use: every call fails loudly if it has not been built or no GPU is present.
"""
