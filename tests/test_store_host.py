"""Host logic without a GPU: the chunk store's row allocator (first-fit
runs, eviction with merging) and the loading controller (a host-only
library call)."""
import types

import torch

from rag_kv_cache_layer_gb300 import api


def _store(rows):
    shape = types.SimpleNamespace(n_layers=2)
    model = types.SimpleNamespace(shape=shape, kvw=4, dtype=torch.float32,
                                  device=torch.device("cpu"))
    return api.ChunkStore(model, rows)


def test_rows_are_reused_first_fit_and_merged():
    st = _store(100)
    a = st._alloc(30); st.where["a"] = (a, 30)
    b = st._alloc(30); st.where["b"] = (b, 30)
    c = st._alloc(30); st.where["c"] = (c, 30)
    assert (a, b, c) == (0, 30, 60) and st.used == 90
    st.evict("b")
    assert st.free == [(30, 30), (90, 10)] and st.used == 60
    d = st._alloc(25); st.where["d"] = (d, 25)
    assert d == 30                       # first fit: the evicted run
    st.evict("a")
    st.evict("c")
    assert st.free == [(0, 30), (55, 45)]
    st.evict("d")
    assert st.free == [(0, 100)] and st.used == 0


def test_store_full_is_an_error():
    st = _store(10)
    st._alloc(8)
    try:
        st._alloc(3)
    except RuntimeError:
        return
    raise AssertionError("allocation past capacity must fail")


def test_loading_controller_picks_the_largest_hidden_ratio():
    """CacheBlend blog, "Hiding Recompute Behind I/O": r = max(r_load, 15%),
    r_load the largest ratio whose per-layer recompute fits in the per-layer
    load time."""
    table = {500: 0.10, 1500: 0.25, 3000: 0.45, 5000: 0.70, 10000: 1.30}
    assert api.loading_controller(0.50, table) == 3000
    assert api.loading_controller(0.05, table) == 1500      # nothing hidden: the floor
    assert api.loading_controller(2.00, table) == 10000
    assert api.loading_controller(0.30, table, min_ratio_bp=2000) == 2000
