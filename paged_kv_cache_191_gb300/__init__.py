"""GB300-native paged-KV decode attention.

The compute path lives in ``libpagedkv.so`` (hand-written sm_103a CUDA
kernels behind a C ABI, declared in ``include/pagedkv.h``).  This package is
the thin Python binding over that library (``ops``) plus the seeded synthetic
input generators (``workloads``).  Importing the package does not load the
library; the first call into ``ops`` does, and raises if it is missing.
"""
__all__ = ["ops", "workloads"]
