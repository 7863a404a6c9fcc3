"""LazyAttention over a paged, position-agnostic KV cache, for one NVIDIA GB300 (sm_103a).

* ``paged_kv_cache_57_gb300.lazy_attn`` -- Python binding of the C ABI in
  ``include/lazy_attn.h`` (loads ``_lib/liblazyattn.so``; raises if it is missing).
* ``paged_kv_cache_57_gb300.workloads`` -- seeded synthetic workloads (Zipf-shared
  documents in 16-token physical blocks).
* ``paged_kv_cache_57_gb300.build`` -- nvcc build of the library.

The binding is imported on first use so that the workload generator and the build
step work on machines without the compiled library.
"""
__all__ = ["lazy_attn", "workloads", "build"]
