"""GB300 (sm_103a) block-scaled FP4 GEMM and quantiser.

The compute lives in ``libqfp4.so`` (CUDA, C ABI declared in ``include/qfp4.h``);
``block_scaled_fp4_tcgen05_gb300.qfp4`` is its thin Python binding.  Importing
this package loads nothing: the library is opened on first use, and every call
fails loudly if it is missing.
"""
MXFP4 = 0
NVFP4 = 1
