"""GB300 (sm_103a) Leyline AMORTIZE splice of a paged MLA KV cache.

The work runs in libleyline.so (C ABI: include/leyline.h); ``leyline`` is its
thin ctypes binding and ``runtime`` holds the pool / block-table helpers that a
caller uses to lay out a paged cache in torch device memory.
"""
from ._build import build  # noqa: F401
from . import leyline  # noqa: F401

__all__ = ["build", "leyline"]
