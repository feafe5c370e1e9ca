"""GB300-native attention over a paged KV cache.

The compute lives in a C-ABI CUDA library (``libpagedkv.so``, built for
sm_103a from ``csrc/``); ``paged_kv_cache_52_gb300.pagedkv`` is the thin ctypes
binding over it.  Importing this package does not load the library, so the
seeded input generators in ``workloads`` stay usable on machines without a
GPU; the binding fails loudly when the library is missing.
"""

__version__ = "0.1.0"
