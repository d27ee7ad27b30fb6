"""CPU oracle for CacheBlend-style blended prefill -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``rag_kv_cache_layer_gb300``) never imports it and has no CPU
fallback.
"""
from .cacheblend import *  # noqa: F401,F403
from .qcfuse import *  # noqa: F401,F403
