"""paged_kv_gqa_14_gb300: paged grouped-query attention and fused RoPE-and-append for GB300.

The compute lives in the CUDA library ``_build/libpkv.so`` (C ABI: ``include/pkv.h``),
built by ``paged_kv_gqa_14_gb300.build``.  ``ops`` is the thin torch binding with the
ABI's names; ``workloads`` draws seeded synthetic batches; ``staging`` lays one step's host
inputs out in one pinned buffer for a single upload.
"""

__all__ = ["ops", "workloads", "build", "staging"]
