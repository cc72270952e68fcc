"""Paged KV-cache attention for one GB300 (sm_103a).

The library is ``libpkv.so`` (hand-written CUDA behind a C ABI, declared in
``include/pkv.h``); ``paged_kv_cache_200_gb300.pkv`` is its thin ctypes
binding.  The binding is loaded on first use so that the input generators in
``workloads`` can be imported without a GPU.
"""

__all__ = ["pkv", "workloads"]
