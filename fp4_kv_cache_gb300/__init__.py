"""CSA2 (Compressed Sparse Attention 2) decode/prefill hot path for GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind the C-ABI library
``libcsa2.so`` (declared in ``include/csa2.h``); ``fp4_kv_cache_gb300.csa2`` is the
thin ctypes binding with the same entry-point names, and
``fp4_kv_cache_gb300.layers`` strings them into the Full / Reindex / Reuse layer
flows.  Importing the package does not load the library; the first call does, and
fails loudly if it is missing.
"""
