"""GB300-native paged KV cache: slot-mapped K/V store and paged decode / chunked-prefill
attention for Llama-3.2-1B-shaped grouped-query attention.

The compute lives in ``libpagedkv.so`` (hand-written sm_103a CUDA behind a C ABI declared
in ``include/pagedkv.h``).  ``paged_kv_cache_299_gb300.binding`` marshals torch tensors to
that ABI; importing this package does not load the library, calling any entry point does,
and a missing library raises instead of falling back to anything else.
"""

__all__ = ["binding", "workloads"]
