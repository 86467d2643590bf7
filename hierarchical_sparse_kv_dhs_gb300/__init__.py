"""GB300-native hierarchical sparse KV resolution + gather.

The product is ``libdhs.so`` (C ABI in include/dhs.h): hand-written sm_103a
kernels for the per-decode-step path of Adaptive DHiSparse -- resolve each
request's top-k selected rows through the tail / optional map, the
B-bounded hot cache with LRU, and pinned host memory, then gather them into
attention staging.  ``dhs`` is its ctypes binding; ``runner`` drives whole
synthetic workloads through it.

Build with ``hierarchical_sparse_kv_dhs_gb300.build.build()``.  Importing
``hierarchical_sparse_kv_dhs_gb300.dhs`` without the built library raises.
"""
