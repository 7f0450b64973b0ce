"""KIVI-style 2/4/8-bit KV cache with a fused decode-attend step for NVIDIA
GB300 (sm_103a): a CUDA library behind the C ABI of include/vq_kivi.h, and a
thin Python binding (``cache.KiviCache``) that passes torch tensor pointers
and the current CUDA stream.

Importing the package loads nothing; ``KiviCache`` loads the compiled
library on first use and raises if it is missing.
"""
__all__ = ["KiviCache", "PLANES"]


def __getattr__(name):
    if name in ("KiviCache", "PLANES"):
        from . import cache
        return getattr(cache, name)
    raise AttributeError(name)
