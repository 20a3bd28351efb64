"""GB300-native partitioned KV cache and attention for streaming VLA inference.

The compute path lives in the CUDA library ``librx.so`` (``csrc/``), reached
through the C ABI declared in ``include/rx.h``; ``partitioned_kv_cache_gb300.rx``
is the thin Python binding.  ``workload`` draws the seeded synthetic inputs.
Importing this package does not load the library; importing ``.rx`` does, and
fails loudly if it has not been built.
"""
__all__ = ["workload", "rx"]
