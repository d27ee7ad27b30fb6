"""Pins of the oracle's query-aware selectors (QCFuse §3.2-3.4) against what
the page and the mathematics fix.  No GPU.

* Eq. 14 anchor counts are ceilings; Sink keeps each chunk's first
  positions; Knorm ranks the lowest key norms first and, since a rotation
  preserves norms, does not depend on where the chunk is placed.
* The attention mass of each (query row, q head) is a softmax over the
  context, so the masses sum to rows x heads; a zero query spreads it evenly;
  q head h reads kv head floor(h / group).
* Eq. 9: with a single chunk, the stitched PIC context equals the full
  prefill's context exactly (causal prefix), so the probe's query rows must
  reproduce the full prefill's rows at every layer.
* RoPE is relative: moving the prefix and the query rows by the same offset
  rotates every probe key by that offset and nothing else.  A probe that used
  any other position ids for the query rows than the ones it is given
  breaks this.
* Eq. 11 endpoints: rho = 1 selects every context position, rho = 0 none;
  with P = C the blend is the full prefill.
"""
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
    assert float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) <= tol * scale


# ------------------------------------------------------------------ anchors
@pytest.mark.parametrize("n,bp,want", [(512, 1000, 52), (10, 1000, 1), (10, 0, 0),
                                       (7, 10000, 7), (3, 3334, 2), (3, 3333, 1),
                                       (400, 1000, 40)])
def test_anchor_count_is_the_ceiling(n, bp, want):
    assert O.anchor_count(n, bp) == want


def test_sink_anchors_are_the_chunk_head():
    assert list(O.anchor_positions(O.sink_anchor_scores(20), 2500)) == [0, 1, 2, 3, 4]


def test_knorm_anchors_lowest_norm_first_ties_to_lower_position():
    # 2 layers x 6 positions x 4 dims; position r's keys are scaled by s[r]
    # in both layers, so its summed squared norm is s[r]^2 * (|a|^2 + |b|^2)
    s = np.array([3.0, 1.0, 2.0, 1.0, 0.5, 4.0])
    a = np.array([1.0, -2.0, 0.5, 1.5])
    b = np.array([0.0, 1.0, -1.0, 2.0])
    K = np.stack([s[:, None] * a[None, :], s[:, None] * b[None, :]])
    # norms in order: 4 (0.25), then 1 and 3 tied (1.0), 2, 0, 5
    assert list(O.anchor_positions(O.knorm_anchor_scores(K), 5000)) == [1, 3, 4]
    assert list(O.anchor_positions(O.knorm_anchor_scores(K), 3333)) == [1, 4]


def test_knorm_scores_do_not_depend_on_the_chunk_offset():
    m = _model()
    chunks, query, segs, store = _request(m)
    k_local = store[1][0]
    moved = np.stack([O.reposition_keys(k_local[l], 37, m.n_kv_heads, m.head_dim, m.rope_base)
                      for l in range(m.n_layers)])
    _close(O.knorm_anchor_scores(moved), O.knorm_anchor_scores(k_local), 1e-12)


# ------------------------------------------------------------ attention mass
def test_attention_mass_sums_to_rows_times_heads():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(5, 4, 8))
    K = rng.normal(size=(11, 2 * 8))
    mass = O.attention_mass(q, K, 4, 2)
    assert mass.shape == (11,) and np.all(mass > 0)
    _close(mass.sum(), 5 * 4, 1e-12)


def test_attention_mass_of_a_zero_query_is_uniform():
    K = np.random.default_rng(4).normal(size=(8, 2 * 6))
    mass = O.attention_mass(np.zeros((3, 4, 6)), K, 4, 2)
    _close(mass, np.full(8, 3 * 4 / 8), 1e-12)


def test_attention_mass_reads_kv_head_of_the_group():
    # kv head 0 has one large key aligned with the queries at t = 1, kv head 1
    # at t = 3; q heads 0, 1 belong to kv head 0 and q heads 2, 3 to kv head 1
    hd = 4
    v = np.array([1.0, 0.0, 0.0, 0.0])
    K = np.zeros((5, 2, hd))
    K[1, 0] = 40 * v
    K[3, 1] = 40 * v
    # only q heads 0 and 1 (kv head 0) look along v; heads 2, 3 are zero and
    # spread their mass evenly, so t = 1 collects about 2 rows x 2 heads and
    # t = 3 only its even share (a head -> kv head map of h % Hkv fails this)
    q = np.tile(v, (2, 4, 1))                       # 2 rows x 4 q heads
    q[:, 2:] = 0.0
    mass = O.attention_mass(q, K.reshape(5, 2 * hd), 4, 2)
    assert mass[1] > 2 * 2 * 0.99
    assert abs(mass[3] - 2 * 2 / 5) < 1e-3


# ------------------------------------------------------------------ probe
def test_full_view_probe_of_one_chunk_is_the_full_prefill():
    m = _model()
    rng = np.random.default_rng(5)
    chunk = rng.integers(0, m.vocab, size=11)
    query = rng.integers(0, m.vocab, size=4)
    full = O.full_prefill(m, np.concatenate([chunk, query]))
    kc, vc = O.chunk_prefill(m, chunk)
    n = len(chunk)
    out = O.probe_query_states(m, query, n + np.arange(len(query)), kc, vc, m.n_layers - 1)
    for l in range(m.n_layers):
        _close(out[l][1], full.K[l, n:], 1e-10)


def test_probe_positions_are_relative():
    m = _model()
    chunks, query, segs, store = _request(m)
    K, V = O.stitch(store, [len(c) for c in chunks], m.n_kv_heads, m.head_dim, m.rope_base)
    N = K.shape[1]
    anchors = np.array([0, 2, 3, 8, 12, 17, 19])
    u_pos = N + np.arange(len(query))
    base = O.probe_query_states(m, query, u_pos, K[:, anchors], V[:, anchors], m.n_layers - 1)
    delta = 29
    Ks = np.stack([O.reposition_keys(K[l][anchors], delta, m.n_kv_heads, m.head_dim,
                                     m.rope_base) for l in range(m.n_layers)])
    moved = O.probe_query_states(m, query, u_pos + delta, Ks, V[:, anchors], m.n_layers - 1)
    for l in range(m.n_layers):
        _close(moved[l][1], O.reposition_keys(base[l][1], delta, m.n_kv_heads, m.head_dim,
                                              m.rope_base), 1e-10)


def test_anchor_probe_differs_from_full_view_but_keeps_the_mass_total():
    m = _model()
    chunks, query, segs, store = _request(m)
    P_full, I_full, a_full = O.query_probe_select(m, segs, store, 3000, "all")
    P_sink, I_sink, a_sink = O.query_probe_select(m, segs, store, 3000, "sink", 2500, [1, 2])
    N = sum(len(c) for c in chunks)
    assert list(a_full) == list(range(N))
    # Sink at 25% keeps ceil(n/4) head positions of each chunk
    assert list(a_sink) == [0, 1, 7, 8, 9, 16, 17]
    _close(I_full.sum(), m.n_layers * len(query) * m.n_q_heads, 1e-10)
    _close(I_sink.sum(), 2 * len(query) * m.n_q_heads, 1e-10)


# ---------------------------------------------------------- selection, blend
def test_query_probe_select_endpoints():
    m = _model()
    chunks, query, segs, store = _request(m)
    N = sum(len(c) for c in chunks)
    assert list(O.query_probe_select(m, segs, store, 10000, "knorm", 1000)[0]) == list(range(N))
    assert len(O.query_probe_select(m, segs, store, 0, "knorm", 1000)[0]) == 0
    P, I, _ = O.query_probe_select(m, segs, store, 3000, "knorm", 3000, [0, 2])
    assert len(P) == O.select_count(N, 3000) and np.all(np.diff(P) > 0)
    assert list(P) == list(O.token_topk(I, len(P)))


def test_query_probe_blend_with_every_position_is_the_full_prefill():
    m = _model()
    chunks, query, segs, store = _request(m)
    res, I, _ = O.query_probe_blend(m, segs, store, 10000, "sink", 5000, [1])
    full = O.full_prefill(m, np.concatenate(chunks + [query]))
    _close(res.K, full.K, 1e-9)
    _close(res.hidden[-1], full.hidden[-1], 1e-9)
    assert res.token == full.token
