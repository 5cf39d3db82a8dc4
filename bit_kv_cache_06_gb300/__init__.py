"""bit_kv_cache_06_gb300 -- KIVI-style 2/4-bit KV-cache quantisation and
decode attention for one GB300 GPU.

The product is libkivi.so (C ABI in include/kivi.h); ``kivi`` is its thin
ctypes binding, ``build`` compiles it with nvcc for sm_103a, and ``synth``
holds the seeded synthetic workloads used by the tests and the benchmark.
"""
from . import kivi  # noqa: F401  (loads the library lazily, on first call)
from .kivi import CacheShape, KiviCache, KiviError  # noqa: F401
