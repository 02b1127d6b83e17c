"""GB300-native DSA lightning-indexer path: paged key store, tcgen05 scoring and
exact top-k, shipped as the C-ABI library libdsaidx.so (include/dsaidx.h).

Submodules:
  dsaidx     -- ctypes binding of the library (argument marshalling only)
  build      -- nvcc build of the library for sm_103a
  workloads  -- seeded synthetic inputs (no arithmetic of the method)
"""
