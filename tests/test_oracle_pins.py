"""Pins of the CPU oracle's primitives against closed forms, hand-derived
values, the pages' printed numbers, brute force and independent library
routines.  No GPU."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import workload as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- RoPE ----
def test_rope_inv_freq_closed_form():
    # theta_e = base^(-2e/hd): hd=4, base=10000 -> [1, 10000^-0.5]
    np.testing.assert_allclose(O.rope_inv_freq(4, 10000.0), [1.0, 0.01],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.rope_inv_freq(8, 16.0),
                               [1.0, 0.5, 0.25, 0.125], rtol=0, atol=0)


def test_rope_hand_value_sign_convention():
    # hd=2: one pair, theta_0 = 1; (1, 0) rotated by angle 1 -> (cos 1, sin 1)
    x = np.array([[[1.0, 0.0]]])
    out = O.rope_rotate(x, np.array([1]), 10000.0)
    np.testing.assert_allclose(out[0, 0], [0.5403023058681398,
                                           0.8414709848078965], atol=1e-15)
    # (0, 1) rotated by angle 1 -> (-sin 1, cos 1)
    out = O.rope_rotate(np.array([[[0.0, 1.0]]]), np.array([1]), 10000.0)
    np.testing.assert_allclose(out[0, 0], [-0.8414709848078965,
                                           0.5403023058681398], atol=1e-15)


def test_rope_matches_complex_rotation():
    # Textbook form of the rotary embedding: pair (x_e, x_{e+hd/2}) is the
    # complex number x_e + i x_{e+hd/2}, multiplied by exp(i pos theta_e).
    rng = np.random.default_rng(0)
    hd, H, n, base = 16, 3, 7, 500.0
    x = rng.standard_normal((n, H, hd))
    pos = rng.integers(0, 40000, size=n)
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    theta = base ** (-np.arange(0, hd, 2) / hd)
    z = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    ref = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(O.rope_rotate(x, pos, base), ref, rtol=1e-12,
                               atol=1e-12)


def test_rope_composition_and_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 2, 64))
    for a, b in [(0, 0), (3, 7), (511, 2560), (30000, 3000)]:
        two = O.rope_rotate(O.rope_rotate(x, a, 1e4), b, 1e4)
        one = O.rope_rotate(x, a + b, 1e4)
        np.testing.assert_allclose(two, one, rtol=1e-9, atol=1e-9)
    assert np.array_equal(O.rope_rotate(x, 0, 1e4), x)      # delta 0: exact
    # each pair keeps its norm
    y = O.rope_rotate(x, 1234, 1e4)
    n0 = x[..., :32] ** 2 + x[..., 32:] ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    np.testing.assert_allclose(n0, n1, rtol=1e-12)


def test_reposition_equals_rotation_at_request_position():
    # keys stored at chunk-local t, moved by delta == keys rotated at t+delta
    rng = np.random.default_rng(2)
    raw = rng.standard_normal((9, 2, 32))
    t = np.arange(9)
    stored = O.rope_rotate(raw, t, 1e4).reshape(9, 64)
    moved = O.reposition_keys(stored, 100, 2, 32, 1e4)
    direct = O.rope_rotate(raw, t + 100, 1e4).reshape(9, 64)
    np.testing.assert_allclose(moved, direct, rtol=1e-10, atol=1e-10)


def test_stitch_offsets_and_values():
    rng = np.random.default_rng(3)
    lens = [3, 5, 2]
    raw = [rng.standard_normal((2, n, 1, 8)) for n in lens]   # 2 layers
    store = []
    for r, n in zip(raw, lens):
        k = np.stack([O.rope_rotate(r[l], np.arange(n), 1e4).reshape(n, 8)
                      for l in range(2)])
        v = rng.standard_normal((2, n, 8))
        store.append((k, v))
    K, V = O.stitch(store, lens, 1, 8, 1e4)
    assert K.shape == (2, 10, 8)
    off = 0
    for (k, v), r, n in zip(store, raw, lens):
        for l in range(2):
            np.testing.assert_allclose(
                K[l, off:off + n],
                O.rope_rotate(r[l], np.arange(off, off + n), 1e4).reshape(n, 8),
                rtol=1e-10, atol=1e-10)
            assert np.array_equal(V[l, off:off + n], v[l])     # V unchanged
        off += n


# ------------------------------------------------------- norm / silu ----
def test_rms_norm_hand_value():
    out = O.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(out[0], [3 / r, 8 / r], rtol=1e-15)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 33))
    g = rng.standard_normal(33)
    ref = F.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-5)
    np.testing.assert_allclose(O.rms_norm(x, g, 1e-5), ref.numpy(), rtol=1e-12)


def test_silu():
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(np.array([1.0])), [0.7310585786300049],
                               rtol=1e-15)
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------- attention ----
def test_attention_hand_value():
    # one head, hd=4, scale 1/2: scores 0 and ln3 -> weights 1/4, 3/4
    q = np.array([[[1.0, 0, 0, 0]], [[1.0, 0, 0, 0]]])
    K = np.array([[[0.0, 0, 0, 0]], [[2 * math.log(3.0), 0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]])
    out = O.causal_attention(q, np.array([1, 0]), K, V, 1, 1)
    np.testing.assert_allclose(out[0, 0], [0.25, 0.75, 0, 0], atol=1e-15)
    np.testing.assert_array_equal(out[1, 0], [1.0, 0, 0, 0])   # only key 0


def test_attention_matches_torch_sdpa_gqa_scattered_queries():
    rng = np.random.default_rng(5)
    T, Hq, Hkv, hd = 50, 6, 2, 16
    K = rng.standard_normal((T, Hkv, hd))
    V = rng.standard_normal((T, Hkv, hd))
    pos = np.sort(rng.choice(T, size=13, replace=False))
    q = rng.standard_normal((13, Hq, hd))
    out = O.causal_attention(q, pos, K, V, Hq, Hkv)
    tq = torch.from_numpy(q).permute(1, 0, 2)                      # [Hq,n,hd]
    tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(3, dim=0)
    tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(3, dim=0)
    allowed = torch.from_numpy(np.arange(T)[None, :] <= pos[:, None])
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10,
                               atol=1e-12)


def test_attention_is_causal():
    rng = np.random.default_rng(6)
    K = rng.standard_normal((20, 1, 8))
    V = rng.standard_normal((20, 1, 8))
    q = rng.standard_normal((3, 2, 8))
    pos = np.array([2, 9, 15])
    a = O.causal_attention(q, pos, K, V, 2, 1)
    K2, V2 = K.copy(), V.copy()
    K2[16:] = 1e3
    V2[16:] = -7
    b = O.causal_attention(q, pos, K2, V2, 2, 1)
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------- decoder layer (torch) ----
def _tiny_model(seed=0, n_layers=1, d=32, Hq=4, Hkv=2, hd=8, F_=24, V=50):
    rng = np.random.default_rng(seed)
    layers = []
    for _ in range(n_layers):
        layers.append({
            "w_qkv": rng.standard_normal(((Hq + 2 * Hkv) * hd, d)) * 0.3,
            "w_o": rng.standard_normal((d, Hq * hd)) * 0.3,
            "w_gate": rng.standard_normal((F_, d)) * 0.3,
            "w_up": rng.standard_normal((F_, d)) * 0.3,
            "w_down": rng.standard_normal((d, F_)) * 0.3,
            "norm1": 1 + 0.1 * rng.standard_normal(d),
            "norm2": 1 + 0.1 * rng.standard_normal(d),
        })
    return O.Model(n_layers, d, Hq, Hkv, hd, F_, V, 10000.0, 1e-5,
                   rng.standard_normal((V, d)), 1 + 0.1 * rng.standard_normal(d),
                   layers)


def _torch_layer(m, L, h, pos):
    """The same decoder block written with torch library routines: F.linear
    (x W^T for W stored [out, in]), F.rms_norm, complex-number rotary
    embedding, scaled_dot_product_attention, F.silu."""
    t = lambda a: torch.from_numpy(np.asarray(a))
    Hq, Hkv, hd = m.n_q_heads, m.n_kv_heads, m.head_dim
    n = h.shape[0]
    h = t(h)
    x = F.rms_norm(h, (m.d_model,), t(L["norm1"]), eps=m.norm_eps)
    wq, wk, wv = torch.split(t(L["w_qkv"]), [Hq * hd, Hkv * hd, Hkv * hd])
    q = F.linear(x, wq).view(n, Hq, hd)
    k = F.linear(x, wk).view(n, Hkv, hd)
    v = F.linear(x, wv).view(n, Hkv, hd)
    theta = m.rope_base ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(n, hd // 2, dtype=torch.float64),
                      t(pos).double()[:, None] * theta[None, :])[:, None, :]

    def rope(a):
        z = torch.complex(a[..., : hd // 2], a[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)
    q, k = rope(q), rope(k)
    g = Hq // Hkv
    o = F.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1).repeat_interleave(g, 0),
        v.transpose(0, 1).repeat_interleave(g, 0), is_causal=True)
    h1 = h + F.linear(o.transpose(0, 1).reshape(n, Hq * hd), t(L["w_o"]))
    x2 = F.rms_norm(h1, (m.d_model,), t(L["norm2"]), eps=m.norm_eps)
    mlp = F.linear(F.silu(F.linear(x2, t(L["w_gate"]))) *
                   F.linear(x2, t(L["w_up"])), t(L["w_down"]))
    return (h1 + mlp).numpy(), k.reshape(n, -1).numpy(), v.reshape(n, -1).numpy()


def test_decoder_layer_matches_torch_composition():
    m = _tiny_model()
    rng = np.random.default_rng(9)
    T = 11
    h = rng.standard_normal((T, m.d_model))
    K = np.zeros((T, m.n_kv_heads * m.head_dim))
    V = np.zeros_like(K)
    rows = np.arange(T)
    h2, k, v = O.decoder_layer(m, 0, h, rows, K, V, rows)
    rh, rk, rv = _torch_layer(m, m.layers[0], h, rows)
    np.testing.assert_allclose(h2, rh, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(k, rk, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(v, rv, rtol=1e-10, atol=1e-10)
    np.testing.assert_array_equal(K, k)     # written into the cache rows


def test_first_token_hand_value():
    m = _tiny_model(V=5)
    m.embed[:] = 0.0
    m.final_norm[:] = 1.0
    h = np.zeros(m.d_model)
    h[3] = 2.0
    m.embed[4, 3] = 1.0
    m.embed[1, 3] = -1.0
    assert O.first_token(m, h) == 4
    m.embed[2, 3] = 1.0            # tie between ids 2 and 4 -> lowest id
    assert O.first_token(m, h) == 2


# ----------------------------------------------------------- selection ----
def test_deviation_hand_value():
    d = O.kv_deviation(np.array([[1.0, 2.0], [0.0, 0.0]]),
                       np.array([[0.0, 0.0], [3.0, 4.0]]))
    np.testing.assert_array_equal(d, [5.0, 25.0])


def test_select_count_golden():
    g = json.load(open(os.path.join(GOLD, "select_count.json")))
    for c in g["cases"]:
        assert O.select_count(c["n_ctx"], c["ratio_bp"]) == c["k"], c


def _brute_topk(d, k):
    """The unique k-subset S where every member beats every non-member
    (larger value, or equal value and lower index)."""
    n = len(d)
    beats = lambda i, j: d[i] > d[j] or (d[i] == d[j] and i < j)
    found = [S for S in itertools.combinations(range(n), k)
             if all(beats(i, j) for i in S for j in range(n) if j not in S)]
    assert len(found) == 1
    return list(found[0])


@pytest.mark.parametrize("n", range(1, 10))
def test_token_topk_brute_force(n):
    rng = np.random.default_rng(n)
    for trial in range(6):
        if trial % 3 == 0:
            d = rng.standard_normal(n) ** 2
        elif trial % 3 == 1:
            d = rng.integers(0, 3, size=n).astype(float)      # many ties
        else:
            d = np.full(n, 1.5)                                # all tied
        for k in range(0, n + 1):
            assert list(O.token_topk(d, k)) == _brute_topk(d, k)


def test_doc_aligned_golden():
    g = json.load(open(os.path.join(GOLD, "doc_aligned.json")))
    for c in g["cases"]:
        got = O.doc_aligned_select(np.array(c["d"], float), c["spans"], c["k"])
        assert list(got) == c["expect"], c


def _doc_aligned_properties_hold(d, offs, k, got):
    """Checks a selection against the statements of "Request Order Matters"
    §2.3 (Eq. 3 and the policy text) one by one, without re-running the
    policy: the result splits into whole spans W and at most one contiguous
    window inside one further span p; W is a prefix of the spans ranked by
    mean deviation (ties: lower span), skipping none that would fit; p is the
    first ranked span after W (the first that does not fit), and the window
    has the largest total deviation among all windows of its length inside p,
    leftmost on ties; exactly k tokens."""
    spans = [(a, b) for a, b in zip(offs[:-1], offs[1:]) if b > a]
    got = set(int(i) for i in got)
    if len(got) != k:
        return False
    whole = [j for j, (a, b) in enumerate(spans) if set(range(a, b)) <= got]
    rest = got - set().union(*[set(range(*spans[j])) for j in whole]) if whole else set(got)
    mean = lambda j: sum(d[spans[j][0]:spans[j][1]]) / (spans[j][1] - spans[j][0])
    ranked = sorted(range(len(spans)), key=lambda j: (-mean(j), j))
    # W is exactly the first len(W) ranked spans
    if sorted(whole) != sorted(ranked[:len(whole)]):
        return False
    if not rest:
        # no window: the budget is used up by whole spans (or k covers everything)
        return sum(spans[j][1] - spans[j][0] for j in whole) == k
    # the window: contiguous, inside the next ranked span, which does not fit whole
    p = ranked[len(whole)]
    a, b = spans[p]
    lo, hi = min(rest), max(rest)
    if not (a <= lo and hi < b and hi - lo + 1 == len(rest)):
        return False
    if b - a <= k - sum(spans[j][1] - spans[j][0] for j in whole):
        return False          # p would have fitted whole
    w = len(rest)
    sums = [sum(d[s:s + w]) for s in range(a, b - w + 1)]
    return sums[lo - a] == max(sums) and sums.index(max(sums)) == lo - a


def test_doc_aligned_random_against_the_policy_statements():
    rng = np.random.default_rng(11)
    for _ in range(200):
        m = rng.integers(1, 6)
        lens = rng.integers(0, 7, size=m)
        offs = [0] + list(np.cumsum(lens))
        N = offs[-1]
        if N == 0:
            continue
        d = rng.integers(0, 5, size=N).astype(float)
        for k in range(0, N + 1):
            got = list(O.doc_aligned_select(d, offs, k))
            assert _doc_aligned_properties_hold(d, offs, k, got), (d, offs, k, got)


def test_doc_aligned_property_check_rejects_wrong_selections():
    # the property check itself: a selection that breaks each statement fails
    d = np.array([5.0, 5, 1, 1, 9, 9, 9, 0], dtype=float)
    offs = [0, 2, 4, 8]        # means 5, 1, 6.75
    assert _doc_aligned_properties_hold(d, offs, 6, [0, 1, 4, 5, 6, 7])
    assert not _doc_aligned_properties_hold(d, offs, 6, [0, 1, 2, 3, 4, 5])   # skips rank 2
    assert _doc_aligned_properties_hold(d, offs, 5, [0, 4, 5, 6, 7])          # tie in span 0: leftmost
    assert not _doc_aligned_properties_hold(d, offs, 5, [1, 4, 5, 6, 7])      # not the leftmost
    assert not _doc_aligned_properties_hold(d, offs, 5, [3, 4, 5, 6, 7])      # window not in the next span
    assert _doc_aligned_properties_hold(d, offs, 3, [4, 5, 6])                # best window of span 2
    assert not _doc_aligned_properties_hold(d, offs, 3, [5, 6, 7])            # not the best window
    assert not _doc_aligned_properties_hold(d, offs, 2, [4])                  # wrong size


def test_doc_aligned_whole_document_budget():
    # k equal to one document's length, that document ranked first -> it alone
    d = np.concatenate([np.full(400, 1.0), np.full(400, 3.0), np.full(400, 2.0)])
    got = O.doc_aligned_select(d, [0, 400, 800, 1200], 400)
    assert list(got) == list(range(400, 800))


# ---------------------------------------------------------- byte model ----
def test_byte_model_matches_printed_numbers():
    g = json.load(open(os.path.join(GOLD, "byte_model.json")))
    for c in g["cases"]:
        b = O.kv_bytes_per_layer(g["context_len"], c["kv_heads"], g["head_dim"])
        assert round(b / 1e6, 1) == c["printed_MB"]
        assert round(b / g["bandwidth_bytes_per_s"] * 1e3, 1) == c["printed_ms"]


# ------------------------------------------------------ Table 2 diagnostics --
def test_selection_segments_by_hand():
    """"Request Order Matters" §4.4 Table 2: segments = separate contiguous
    regions.  Counted by hand: {} none; {3} one; {1,2,3 | 7,8 | 10} three;
    a single 400-token window one."""
    assert O.selection_segments([]) == 0
    assert O.selection_segments([3]) == 1
    assert O.selection_segments([1, 2, 3, 7, 8, 10]) == 3
    assert O.selection_segments(list(range(400, 800))) == 1
    assert O.selection_segments([0, 2, 4, 6]) == 4


def test_captured_deviation_by_hand():
    """Same table: the selected tokens' share of the total deviation.
    d = (1, 2, 3, 4): P = {1, 3} carries (2 + 4) / 10; all of it is 1; the
    top-1 token carries 0.4."""
    d = [1.0, 2.0, 3.0, 4.0]
    assert O.captured_deviation([1, 3], d) == 0.6
    assert O.captured_deviation([0, 1, 2, 3], d) == 1.0
    assert O.captured_deviation([3], d) == 0.4
    assert O.captured_deviation([], d) == 0.0


def test_kv_rows_is_the_cache_part_of_the_projection():
    """kv_rows gives the k and v of qkv_rows (the same definition without
    the query heads): checked against the fused projection on random rows."""
    shape = W.ModelShape("t", 1, 48, 4, 2, 12, 40, 97, dtype="f32")
    m = O.model_from_weights(shape, W.make_weights(shape, 3, std=0.2))
    h = np.random.default_rng(1).standard_normal((9, 48))
    pos = np.array([0, 1, 5, 7, 30, 31, 100, 101, 4000])
    _, k, v = O.qkv_rows(m, 0, h, pos)
    k2, v2 = O.kv_rows(m, 0, h, pos)
    assert np.allclose(k, k2, rtol=0, atol=1e-12) and np.allclose(v, v2, rtol=0, atol=1e-12)


# ------------------------------------------------- span-policy controls --
def test_single_window_is_doc_aligned_over_one_span():
    """"Request Order Matters" §2.3: single-window is the k-token window of
    largest total deviation -- the document-aligned rule with the whole
    reusable prompt as its only span (k < N takes the window fill)."""
    rng = np.random.default_rng(5)
    for n in range(1, 12):
        for k in range(0, n):
            d = rng.integers(0, 4, size=n).astype(np.float64)     # ties included
            assert list(O.single_window_select(d, k)) == list(O.doc_aligned_select(d, [0, n], k))
    assert list(O.single_window_select(np.array([1., 5., 1., 5., 1.]), 2)) == [0, 1]   # leftmost
    assert list(O.single_window_select(np.array([0., 0., 3., 4., 0.]), 2)) == [2, 3]
    assert list(O.single_window_select(np.array([1., 2.]), 5)) == [0, 1]


def test_fixed_chunk_offsets_by_hand():
    """Same page §4.4: equal spans shifted so they cross document boundaries."""
    assert O.fixed_chunk_offsets(10, 4, 2) == [0, 2, 6, 10]
    assert O.fixed_chunk_offsets(10, 4, 0) == [0, 4, 8, 10]
    assert O.fixed_chunk_offsets(8, 4, 4) == [0, 4, 8]
    assert O.fixed_chunk_offsets(3, 4, 2) == [0, 2, 3]


def test_random_document_order_by_hand():
    """Same page §2.3: random-document keeps the document spans and the fill
    rule but visits spans in a caller-drawn order.  d = 1,1,1 | 5,5,5 |
    2,2,2 with k = 4: visiting (0, 2, 1) takes span 0 whole, then one token
    of span 2 (all equal: leftmost); ranking by mean takes span 1, then
    span 2's first token."""
    d = np.array([1., 1., 1., 5., 5., 5., 2., 2., 2.])
    offs = [0, 3, 6, 9]
    assert list(O.doc_aligned_select(d, offs, 4, order=[0, 2, 1])) == [0, 1, 2, 6]
    assert list(O.doc_aligned_select(d, offs, 4)) == [3, 4, 5, 6]
    # the mean ranking given explicitly reproduces the default
    assert list(O.doc_aligned_select(d, offs, 4, order=[1, 2, 0])) == [3, 4, 5, 6]


def test_first_tokens_by_hand():
    """EPIC's chunk-boundary rule as the QCFuse page describes it (§2): the
    first tokens of every chunk.  Chunks of 5, 4, 6 tokens with k = 7 share
    3, 2, 2; chunks of 2 and 8 with k = 6 share 3, 3, and the short first
    chunk hands its missing token to the second."""
    assert list(O.first_tokens_select([0, 5, 9, 15], 7)) == [0, 1, 2, 5, 6, 9, 10]
    assert list(O.first_tokens_select([0, 2, 10], 6)) == [0, 1, 2, 3, 4, 5]
    assert list(O.first_tokens_select([0, 3, 3, 6], 2)) == [0, 3]          # empty span skipped
    assert list(O.first_tokens_select([0, 4], 9)) == [0, 1, 2, 3]          # k > N
    assert len(O.first_tokens_select([0, 400, 800, 1200], 60)) == 60
