"""B300 (sm_103a) hot path of CSA2 over an FP4 main-KV cache.

The compute lives in libcsa2.so (hand-written CUDA, C ABI in
include/csa2.h); :mod:`fp4_kv_cache_06_b300.csa2` is a thin ctypes binding
with the same names. Importing this package does not load the library; the
binding loads it on first use and raises if it is missing (there is no CPU
fallback).
"""
__all__ = ["csa2"]
