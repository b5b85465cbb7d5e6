"""GB300-native KV residency path for index-based sparse attention (single-GPU DP mode).

``ula`` is the ctypes binding of the C ABI (include/ula.h) implemented by the
CUDA library ``_build/libula.so``; ``cache.UlaCache`` adds the PyTorch pools
and streams.  Build with ``serving_step_sparse_gb300.build.build()``.
"""
__all__ = ["ula", "cache"]
