"""GQA attention over a preallocated KV cache, native to GB300 (sm_103a).

The compute path is the C-ABI library ``libkvc.so`` built from ``csrc/``
(declared in ``include/kvc.h``); this package only marshals arguments to it.
There is no CPU fallback: calls raise if the library is missing.
``workloads`` holds the seeded synthetic input generators.
"""

from ._lib import KVCError, LIB_PATH, lib  # noqa: F401
from .cache import KVCache, PagedKVCache, gqa_attention  # noqa: F401

__all__ = ["KVCache", "PagedKVCache", "KVCError", "gqa_attention", "lib", "LIB_PATH"]
