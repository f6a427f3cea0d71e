"""Fused tensor-parallel matmul + collective operators for GB300 (sm_103a).

The operators run in hand-written CUDA kernels behind a C ABI (``include/coc.h``,
``libcoc.so``); ``coc`` is the thin Python binding over it.
"""
