"""GB300-native paged KV cache hot path: kv_store + paged decode attention.

The compute lives in ``libpkv.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/pkv.h``); :mod:`paged_kv_cache_62_gb300.pkv` is the
thin ctypes binding with the same names.  :mod:`.workloads` builds the seeded
synthetic inputs used by the tests and the benchmark.
"""
__all__ = ["pkv", "workloads"]
