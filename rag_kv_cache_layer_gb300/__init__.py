"""GB300 (sm_103a) CacheBlend-style blended prefill.

The C ABI lives in ``include/cacheblend.h`` and ``libcacheblend.so`` (built
in-tree by ``rag_kv_cache_layer_gb300.build``); ``api`` mirrors it for torch
tensors.  Importing the package fails if the library has not been built.
"""
from . import _lib  # noqa: F401  (loads libcacheblend.so or raises)
from .api import *  # noqa: F401,F403
