"""dense_gemm_10_gb300: a GB300-native dense GEMM, C = alpha * op(A) * op(B) + beta * C.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/gemm_gb300.h``); ``gemm`` is its thin
ctypes binding.  Importing the package loads nothing: the library is opened on
first use, and every call fails loudly if it has not been built.
"""
__all__ = ["gemm", "inputs", "metrics"]
