"""Pins of the oracle's prefill and blend paths against what the pages fix:
the rho = 1 and rho = 0 endpoints (QCFuse §4.1.5), exact reuse of a chunk at
position 0 and the context independence of layer 0 (QCFuse Eqs. 3-5),
causality, and the Eq. 7 fusion rule.  No GPU."""
import numpy as np
import pytest

import oracle as O
import workload as W


def _model(n_layers=3, d=48, Hq=4, Hkv=2, hd=12, F_=40, V=97, seed=0):
    shape = W.ModelShape("t", n_layers, d, Hq, Hkv, hd, F_, V, dtype="f32")
    w = W.make_weights(shape, seed, std=0.15, embed_std=1.0)
    return O.model_from_weights(shape, w)


def _request(m, seed=1, lens=(7, 9, 5), n_query=4):
    rng = np.random.default_rng(seed)
    chunks = [rng.integers(0, m.vocab, size=n) for n in lens]
    query = rng.integers(0, m.vocab, size=n_query)
    segs = [(c, True) for c in chunks] + [(query, False)]
    store = [O.chunk_prefill(m, c) for c in chunks]
    return chunks, query, segs, store


def _close(a, b, tol=1e-10):
    scale = max(1.0, float(np.max(np.abs(b))))
    assert float(np.max(np.abs(a - b))) <= tol * scale


def test_full_prefill_is_causal():
    m = _model()
    toks = np.random.default_rng(2).integers(0, m.vocab, size=20)
    a = O.full_prefill(m, toks)
    b = O.full_prefill(m, toks[:13])
    _close(a.K[:, :13], b.K)
    _close(a.V[:, :13], b.V)
    _close(a.hidden[:13], b.hidden)


def test_chunk_at_position_zero_reuses_exactly():
    m = _model()
    chunks, query, segs, store = _request(m)
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    n0 = len(chunks[0])
    _close(full.K[:, :n0], store[0][0], 1e-12)
    _close(full.V[:, :n0], store[0][1], 1e-12)


def test_layer0_kv_is_context_independent():
    # the layer-0 input is the embedding alone, so fresh layer-0 K equals the
    # re-positioned PIC key and fresh V the stored V, for every chunk
    m = _model()
    chunks, query, segs, store = _request(m)
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    K, V = O.stitch(store, [len(c) for c in chunks], m.n_kv_heads, m.head_dim,
                    m.rope_base)
    N = sum(len(c) for c in chunks)
    _close(full.K[0, :N], K[0])
    _close(full.V[0, :N], V[0])
    # ... but not at layer 1, where cross-chunk attention has acted (Eq. 5)
    assert np.max(np.abs(full.K[1, len(chunks[0]):N] -
                         K[1, len(chunks[0]):])) > 1e-3


def test_full_recompute_equals_full_prefill():
    m = _model()
    chunks, query, segs, store = _request(m)
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    r = O.blend_prefill(m, segs, store, ratio_bp=10000)
    N = sum(len(c) for c in chunks)
    assert list(r.selected) == list(range(N))
    _close(r.K, full.K)
    _close(r.V, full.V)
    _close(r.hidden, full.hidden)
    assert r.token == full.token


def test_zero_recompute_is_direct_reuse():
    # rho = 0: every context entry at layers >= s is the stitched PIC entry
    # and the query is prefilled over KV^PIC(C) (layer 0 is recomputed in
    # full, which reproduces the PIC entries up to rounding)
    m = _model()
    chunks, query, segs, store = _request(m)
    r = O.blend_prefill(m, segs, store, ratio_bp=0)
    assert len(r.selected) == 0
    lens = [len(c) for c in chunks]
    N = sum(lens)
    K, V = O.stitch(store, lens, m.n_kv_heads, m.head_dim, m.rope_base)
    for l in range(1, m.n_layers):
        assert np.array_equal(r.K[l, :N], K[l])
        assert np.array_equal(r.V[l, :N], V[l])
    # independent composition: query rows prefilled over the stitched cache
    T = N + len(query)
    Kc = np.concatenate([K, np.zeros((m.n_layers, len(query), K.shape[2]))], 1)
    Vc = np.concatenate([V, np.zeros_like(Kc[:, N:])], 1)
    qrows = np.arange(N, T)
    h = O.embed_rows(m, query)
    for l in range(m.n_layers):
        h, _, _ = O.decoder_layer(m, l, h, qrows, Kc[l], Vc[l], qrows)
    _close(r.hidden, h, 1e-9)
    for l in range(m.n_layers):
        _close(r.K[l, N:], Kc[l, N:], 1e-9)
    assert r.token == O.first_token(m, h[-1])


def test_first_chunk_has_zero_deviation():
    # chunk 1's causal prefix is the same standalone and in the request
    m = _model()
    chunks, query, segs, store = _request(m)
    r = O.blend_prefill(m, segs, store, ratio_bp=2000)
    n0 = len(chunks[0])
    assert np.all(r.deviation >= 0)
    assert np.max(r.deviation[:n0]) < 1e-18 * max(1.0, np.max(r.deviation))
    assert np.min(r.deviation[n0:]) > 0


def test_selection_at_layer0_sees_no_deviation():
    # at layer 0 the fresh keys equal the re-positioned PIC keys for every
    # chunk, which pins the per-chunk offsets used by the blend's stitching
    m = _model()
    chunks, query, segs, store = _request(m)
    r = O.blend_prefill(m, segs, store, ratio_bp=1500, sel_layer=0)
    assert np.max(r.deviation) < 1e-18


def test_fusion_rule_eq7():
    m = _model()
    chunks, query, segs, store = _request(m)
    r = O.blend_prefill(m, segs, store, ratio_bp=3000)
    lens = [len(c) for c in chunks]
    N = sum(lens)
    k = O.select_count(N, 3000)
    assert len(r.selected) == k
    assert np.all(np.diff(r.selected) > 0)
    assert list(r.selected) == list(O.token_topk(r.deviation, k))
    K, V = O.stitch(store, lens, m.n_kv_heads, m.head_dim, m.rope_base)
    unsel = np.setdiff1d(np.arange(N), r.selected)
    for l in range(1, m.n_layers):
        assert np.array_equal(r.K[l, unsel], K[l, unsel])      # PIC kept
        assert np.array_equal(r.V[l, unsel], V[l, unsel])
        assert np.all(np.abs(r.K[l, r.selected] - K[l, r.selected]).max(1) > 0)
    assert list(r.rows) == list(r.selected) + list(range(N, N + len(query)))


def test_forced_selection_reproduces_free_selection():
    m = _model()
    chunks, query, segs, store = _request(m)
    a = O.blend_prefill(m, segs, store, ratio_bp=2500)
    b = O.blend_prefill(m, segs, store, ratio_bp=2500, forced=a.selected)
    assert np.array_equal(a.K, b.K) and np.array_equal(a.hidden, b.hidden)


def test_gradual_filtering_only_shrinks():
    m = _model(n_layers=4)
    chunks, query, segs, store = _request(m)
    N = sum(len(c) for c in chunks)
    r = O.blend_prefill(m, segs, store, ratio_bp=2000,
                        schedule=[(2, 3), (3, 2)])
    p1, p2, p3 = (set(r.selected_per_layer[l]) for l in (1, 2, 3))
    assert len(p1) == O.select_count(N, 2000) and len(p2) == 3 and len(p3) == 2
    assert p3 <= p2 <= p1


def test_gradual_keep_at_least_current_count_changes_nothing():
    m = _model(n_layers=4)
    chunks, query, segs, store = _request(m)
    a = O.blend_prefill(m, segs, store, ratio_bp=2000)
    b = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=[(2, 10 ** 6), (3, 10 ** 6)])
    assert np.array_equal(a.K, b.K) and np.array_equal(a.hidden, b.hidden)
    assert np.array_equal(a.selected, b.selected)


def test_gradual_step_reranks_the_current_set_by_its_fresh_keys():
    """CacheBlend blog, "The Chicken-and-Egg Problem" (select_hkvd): at a
    filtering layer the rows still selected are ranked again by how far
    their fresh keys of that layer deviate from the reused keys, and the
    largest deviations are kept.  The hidden states entering that layer are
    taken from the same blend truncated just below it."""
    m = _model(n_layers=4)
    chunks, query, segs, store = _request(m)
    Hkv, hd = m.n_kv_heads, m.head_dim
    r = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=[(2, 3)])
    cut = O.Model(2, m.d_model, m.n_q_heads, Hkv, hd, m.d_ffn, m.vocab, m.rope_base,
                  m.norm_eps, m.embed, m.final_norm, m.layers[:2])
    u = O.blend_prefill(cut, segs, [(k[:2], v[:2]) for k, v in store], ratio_bp=2000)
    P = u.selected
    assert np.array_equal(P, r.selected_per_layer[1])
    # fresh layer-2 keys of the selected rows, rotated at their positions
    lw = m.layers[2]
    h = u.hidden[np.searchsorted(u.rows, P)]
    x = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + m.norm_eps) * lw["norm1"]
    qd = m.n_q_heads * hd
    kf = O.rope_rotate((x @ lw["w_qkv"][qd:qd + Hkv * hd].T).reshape(-1, Hkv, hd), P,
                       m.rope_base).reshape(len(P), -1)
    # reused layer-2 keys: every chunk's stored keys moved to its offset
    offs = np.concatenate([[0], np.cumsum([len(c) for c in chunks])])
    kr = np.concatenate([O.reposition_keys(k[2], int(o), Hkv, hd, m.rope_base)
                         for (k, _), o in zip(store, offs[:-1])])[P]
    d = ((kf - kr) ** 2).sum(axis=1)
    order = sorted(range(len(P)), key=lambda i: (-d[i], i))[:3]
    assert list(r.selected_per_layer[2]) == sorted(P[order].tolist())
    assert list(r.selected) == sorted(P[order].tolist())


def test_chunk_prefill_all_equals_each_chunk_alone():
    # the layer-outer order of the batched chunk prefill changes nothing
    m = _model()
    chunks, query, segs, store = _request(m)
    for (k, v), (k1, v1) in zip(O.chunk_prefill_all(m, chunks), store):
        assert np.array_equal(k, k1) and np.array_equal(v, v1)


def test_forced_steps_reproduce_the_free_steps():
    m = _model(n_layers=4)
    chunks, query, segs, store = _request(m)
    sch = [(2, 3), (3, 2)]
    a = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=sch)
    b = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=sch, forced=a.selected_per_layer[1],
                        forced_steps={l: a.selected_per_layer[l] for l, _ in sch})
    assert np.array_equal(a.K, b.K) and np.array_equal(a.hidden, b.hidden)
    assert all(np.array_equal(a.selected_per_layer[l], b.selected_per_layer[l]) for l in (1, 2, 3))


def test_forced_step_computes_the_given_rows_from_its_layer_on():
    """A forced step keeps exactly the given rows: from that layer on the
    dropped rows keep the stitched cache (Eq. 7) and the kept ones are
    recomputed, whatever their deviation rank."""
    m = _model(n_layers=4)
    chunks, query, segs, store = _request(m)
    a = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=[(2, 3)])
    P1 = a.selected_per_layer[1]
    d = a.deviation_per_layer[2]
    low = np.sort(sorted(P1.tolist(), key=lambda i: (d[i], i))[:3])   # the smallest deviations
    assert not np.array_equal(low, a.selected_per_layer[2])
    b = O.blend_prefill(m, segs, store, ratio_bp=2000, schedule=[(2, 3)], forced_steps={2: low})
    assert np.array_equal(b.selected_per_layer[2], low) and np.array_equal(b.selected, low)
    K, V = O.stitch(store, [len(c) for c in chunks], m.n_kv_heads, m.head_dim, m.rope_base)
    dropped = np.setdiff1d(P1, low)
    for l in (2, 3):
        assert np.array_equal(b.K[l, dropped], K[l, dropped])
        assert np.array_equal(b.V[l, dropped], V[l, dropped])
        assert np.all(np.abs(b.K[l, low] - K[l, low]).max(1) > 0)
    N = sum(len(c) for c in chunks)
    assert list(b.rows) == list(low) + list(range(N, N + len(query)))


def test_selection_past_last_layer_is_full_prefill():
    m = _model()
    chunks, query, segs, store = _request(m)
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    r = O.blend_prefill(m, segs, store, ratio_bp=1500, sel_layer=m.n_layers)
    _close(r.K, full.K)
    assert r.token == full.token


def test_doc_aligned_policy_in_blend():
    m = _model()
    chunks, query, segs, store = _request(m, lens=(6, 6, 6))
    r = O.blend_prefill(m, segs, store, ratio_bp=3400, policy="doc_aligned")
    k = O.select_count(18, 3400)          # 6
    assert len(r.selected) == k
    ref = O.doc_aligned_select(r.deviation, [0, 6, 12, 18], k)
    assert list(r.selected) == list(ref)


@pytest.mark.slow
def test_tiny_workload_runs():
    wl = W.tiny_blend()
    m = O.model_from_weights(wl.model, W.make_weights(wl.model, wl.seed))
    req = wl.requests[0]
    store = [O.chunk_prefill(m, s.tokens) for s in req.segments if s.cached]
    segs = [(s.tokens, s.cached) for s in req.segments]
    r = O.blend_prefill(m, segs, store, wl.ratio_bp)
    assert len(r.selected) == 57 and r.hidden.shape == (89, 256)


# ------------------------------------------------------------ write-back --
def test_write_back_of_a_full_recompute_is_the_full_prefill_cache():
    """With every context token recomputed (rho = 1) the fused cache is the
    full prefill's, so writing it back stores each chunk's full-prefill K/V
    moved to position 0; re-stitching that store at the same offsets gives
    the full prefill's cache again (rotations compose, QCFuse Eq. 4)."""
    m = _model()
    chunks, query, segs, store = _request(m)
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    r = O.blend_prefill(m, segs, store, ratio_bp=10000)
    new = O.write_back(r, segs, m)
    K, V = O.stitch(new, [len(c) for c in chunks], m.n_kv_heads, m.head_dim, m.rope_base)
    N = sum(len(c) for c in chunks)
    _close(K, full.K[:, :N], 1e-10)
    _close(V, full.V[:, :N], 1e-12)


def test_write_back_without_recompute_keeps_the_store():
    """rho = 0 above layer 0: the fused cache of every layer >= 1 is the
    stitched store, so write-back returns the stored caches there (up to
    the rotation round trip); layer 0 (always recomputed) is the chunk's
    own context-free layer-0 K/V, also unchanged."""
    m = _model()
    chunks, query, segs, store = _request(m)
    r = O.blend_prefill(m, segs, store, ratio_bp=0)
    new = O.write_back(r, segs, m)
    for (k0, v0), (k1, v1) in zip(store, new):
        _close(k1, k0, 1e-10)
        _close(v1, v0, 1e-12)


def test_write_back_makes_the_store_depend_on_history():
    """"Request Order Matters" §4.2: the same chunk's stored caches differ
    after it was reused behind different predecessors."""
    m = _model()
    chunks, query, segs, store = _request(m)
    a = O.write_back(O.blend_prefill(m, segs, store, ratio_bp=5000), segs, m)
    segs2 = [segs[1], segs[0], segs[2], segs[3]]
    store2 = [store[1], store[0], store[2]]
    b = O.write_back(O.blend_prefill(m, segs2, store2, ratio_bp=5000), segs2, m)
    # chunk 1 was first in the second request: its layer >= 1 caches differ
    assert np.abs(a[1][0][1:] - b[0][0][1:]).max() > 1e-6
