"""B300-native (sm_103a) CSA2 hot path: FP4 main-KV caching, indexer Top-K, the hierarchical
candidate pool and sparse attention, behind the C ABI in include/csa2.h.

Submodules:
  csa2   -- thin ctypes binding of libcsa2.so (raises ImportError if the library is not built)
  synth  -- seeded synthetic workloads
  step   -- the decode / prefill steps as sequences of C-ABI calls
"""
