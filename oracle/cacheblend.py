"""Plain, slow, fp64 CPU oracle of non-prefix KV-cache fusion for RAG prefill.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg, never by the CUDA product path.  It shares
no code with the CUDA path (no kernels, headers, tables or helpers); the two
meet only at the seeded inputs of ``workload.py``.

Everything here is float64 numpy.  Library primitives used as single steps:
``@`` (matmul), ``np.exp``, ``np.cos``/``np.sin``, ``np.argsort``/``sorted``.
No blocking, fusion or reordering beyond the definitions cited per function.

Sources ("pages"):
* QCFuse: Query-Aware Cache Fusion via Compressed View for Efficient RAG
  Serving (arxiv 2606.05875) -- Tables 1-2, Eqs. 1-7 and 8-20.
* CacheBlend: Reusing KV Caches When Your Text Isn't a Prefix (blog) --
  "Quantifying the Damage", "Selective Recompute Without Skipping", "The
  Chicken-and-Egg Problem", "Hiding Recompute Behind I/O".
* Request Order Matters: Cache-History Sensitivity in Selective KV-Cache
  Reuse for Rolling Agents -- §2.2 Eqs. 1-2, §2.3 Eq. 3, §4.4.

Readings taken where the pages are silent (each is pinned by a test in
``tests/test_oracle_*.py``):
* decoder block: pre-norm Llama-style (RMSNorm, GQA attention with
  rotate-half RoPE, SwiGLU), no biases, LM head tied to the embedding;
* selection layer s = 1 (0-based) by default; layers < s run in full;
* k = floor(N * r_bp / 10000), at least 1 when r_bp > 0, 0 when r_bp == 0;
* top-k ties: larger deviation first, then lower index; output ascending;
* deviation: squared L2 of post-RoPE keys over all kv heads (Eq. 1 of the
  rolling-agent page); at the selection layer the fused cache follows Eq. 7;
* uncached segments (the query, a new document) are recomputed at every
  layer and are not counted in N.

Parity unpinned: none of the functions below -- every one has a pin in
``tests/test_oracle_pins.py`` or ``tests/test_oracle_blend.py``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Model", "model_from_weights", "rope_inv_freq", "rope_rotate",
    "reposition_keys", "stitch", "rms_norm", "silu", "causal_attention",
    "qkv_rows", "kv_rows", "decoder_layer", "full_prefill", "chunk_prefill",
    "chunk_prefill_all", "kv_deviation",
    "select_count", "token_topk", "doc_aligned_select", "blend_prefill",
    "first_token", "first_token_logits", "embed_rows", "kv_bytes_per_layer",
    "selection_segments", "captured_deviation", "single_window_select",
    "fixed_chunk_offsets", "first_tokens_select", "write_back",
    "BlendResult", "PrefillResult",
]


# --------------------------------------------------------------------------
# model container
# --------------------------------------------------------------------------
@dataclass
class Model:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    rope_base: float
    norm_eps: float
    embed: np.ndarray          # [V, d]
    final_norm: np.ndarray     # [d]
    layers: list               # list of dicts of float64 arrays


def model_from_weights(shape, weights) -> Model:
    """Wrap generator output (float32 arrays) as float64 arrays.  The
    embedding stays in its given (exact) float32 form and is widened to
    float64 row by row where it is used, so a 128K-entry vocabulary does not
    need a float64 copy."""
    f = lambda a: np.asarray(a, dtype=np.float64)
    layers = [{k: f(v) for k, v in lw.items()} for lw in weights["layers"]]
    return Model(shape.n_layers, shape.d_model, shape.n_q_heads,
                 shape.n_kv_heads, shape.head_dim, shape.d_ffn, shape.vocab,
                 float(shape.rope_base), float(shape.norm_eps),
                 weights["embed"], f(weights["final_norm"]), layers)


def embed_rows(m: Model, tokens) -> np.ndarray:
    """h = E[tokens] as float64 (the embedding lookup)."""
    return np.asarray(m.embed[np.asarray(tokens)], dtype=np.float64)


# --------------------------------------------------------------------------
# rotary position embedding and re-positioning
# --------------------------------------------------------------------------
def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """theta_e = base^(-2e/hd), e = 0 .. hd/2-1 (rotary embedding of Su et
    al., the position-encoding scheme the QCFuse page's Eq. 4 remaps)."""
    e = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * e / head_dim)


def rope_rotate(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate-half RoPE of x [n, H, hd] at positions pos [n] (or a scalar).

    Pair (x_e, x_{e+hd/2}) is rotated by the angle pos * theta_e:
        out_e        = x_e cos - x_{e+hd/2} sin
        out_{e+hd/2} = x_{e+hd/2} cos + x_e sin
    """
    hd = x.shape[-1]
    half = hd // 2
    ang = np.multiply.outer(np.asarray(pos, dtype=np.float64),
                            rope_inv_freq(hd, base))           # [n, hd/2]
    c = np.cos(ang)[..., None, :]
    s = np.sin(ang)[..., None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def reposition_keys(k_local: np.ndarray, delta: int, n_kv_heads: int,
                    head_dim: int, base: float) -> np.ndarray:
    """Pi_i of QCFuse Eq. 4 for keys: a chunk prefilled standalone holds keys
    rotated to chunk-local positions t; moving it to request offset
    o = delta applies one more rotation by delta (RoPE rotations compose,
    CacheBlend blog "Why You Can't Just Concatenate").  k_local [n, Hkv*hd]."""
    n = k_local.shape[0]
    k = k_local.reshape(n, n_kv_heads, head_dim)
    return rope_rotate(k, delta, base).reshape(n, n_kv_heads * head_dim)


def stitch(store, lens, n_kv_heads, head_dim, base):
    """KV^PIC(C) = [Pi_1(KV_1); ...; Pi_m(KV_m)] (QCFuse Eq. 4).

    store: list over chunks of (K, V), each [n_layers][len][Hkv*hd];
    returns (K, V) each [n_layers][N][Hkv*hd] with chunk i at offset
    o_i = sum_{j<i} |c_j|; values are stitched in token order unchanged."""
    n_layers = store[0][0].shape[0]
    Ks, Vs = [], []
    for l in range(n_layers):
        off = 0
        kl, vl = [], []
        for (kc, vc), ln in zip(store, lens):
            kl.append(reposition_keys(kc[l], off, n_kv_heads, head_dim, base))
            vl.append(vc[l].copy())
            off += ln
        Ks.append(np.concatenate(kl, 0))
        Vs.append(np.concatenate(vl, 0))
    return np.stack(Ks), np.stack(Vs)


# --------------------------------------------------------------------------
# decoder block pieces
# --------------------------------------------------------------------------
def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g, per row."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def causal_attention(q, q_pos, K, V, n_q_heads, n_kv_heads):
    """softmax(q K^T / sqrt(hd) + causal mask) V for selected query rows.

    q [n, Hq, hd] at positions q_pos [n]; K, V [T, Hkv, hd] hold the cache at
    positions 0..T-1.  A query at position p sees keys 0..p only (QCFuse
    §2.1.3: recomputation stays causal over the partially fused prefix); q head h
    uses kv head floor(h / (Hq/Hkv)) (grouped-query attention).  Attention
    cost is n x T, not T x T (CacheBlend blog, step 4 of blend_layer)."""
    n, Hq, hd = q.shape
    T = K.shape[0]
    group = n_q_heads // n_kv_heads
    q_pos = np.asarray(q_pos)
    mask = np.arange(T)[None, :] > q_pos[:, None]                   # [n, T]
    out = np.empty_like(q)
    for h in range(Hq):
        kh = h // group
        s = (q[:, h, :] @ K[:, kh, :].T) / math.sqrt(hd)            # [n, T]
        s = np.where(mask, -np.inf, s)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, kh, :]
    return out


def qkv_rows(m: Model, l: int, h_rows, pos_rows):
    """The attention inputs of layer l for the rows ``h_rows`` [n, d] at
    request positions ``pos_rows``: x = RMSNorm(h; norm1), then q, k, v =
    x W_q^T, x W_k^T, x W_v^T with q and k rotated at their positions.
    Returns q [n, Hq, hd] and the cache rows k, v [n, Hkv*hd]."""
    L = m.layers[l]
    n = h_rows.shape[0]
    Hq, Hkv, hd = m.n_q_heads, m.n_kv_heads, m.head_dim
    x = rms_norm(h_rows, L["norm1"], m.norm_eps)
    qkv = x @ L["w_qkv"].T
    q = qkv[:, :Hq * hd].reshape(n, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(n, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(n, Hkv, hd)
    q = rope_rotate(q, pos_rows, m.rope_base)
    k = rope_rotate(k, pos_rows, m.rope_base)
    return q, k.reshape(n, Hkv * hd), v.reshape(n, Hkv * hd)


def kv_rows(m: Model, l: int, h_rows, pos_rows):
    """The cache rows of layer l alone: x = RMSNorm(h; norm1), k = x W_k^T
    rotated at the rows' positions and v = x W_v^T ([n, Hkv*hd] each)."""
    L = m.layers[l]
    n = h_rows.shape[0]
    Hq, Hkv, hd = m.n_q_heads, m.n_kv_heads, m.head_dim
    x = rms_norm(h_rows, L["norm1"], m.norm_eps)
    k = x @ L["w_qkv"][Hq * hd:(Hq + Hkv) * hd].T
    v = x @ L["w_qkv"][(Hq + Hkv) * hd:].T
    k = rope_rotate(k.reshape(n, Hkv, hd), pos_rows, m.rope_base)
    return k.reshape(n, Hkv * hd), v


def decoder_layer(m: Model, l: int, h_rows, pos_rows, K_cache, V_cache,
                  cache_rows, write_kv=True):
    """One pre-norm decoder layer for the rows ``h_rows`` [n, d] at request
    positions ``pos_rows``; their fresh K/V are written into the layer's
    cache at ``cache_rows`` (Eq. 7: selected entries replace the reused
    ones) and the rows then attend causally over the whole cache.  Returns
    the new hidden rows and the fresh (post-RoPE) K and V rows.

        x  = RMSNorm(h; norm1)
        q, k, v = x W_q^T, x W_k^T, x W_v^T ; q, k rotated at their positions
        h1 = h + Attn(q, K_fused, V_fused) W_o^T
        h2 = h1 + (silu(x2 W_gate^T) * (x2 W_up^T)) W_down^T, x2 = RMSNorm(h1)
    """
    L = m.layers[l]
    n = h_rows.shape[0]
    Hq, Hkv, hd = m.n_q_heads, m.n_kv_heads, m.head_dim
    q, k_new, v_new = qkv_rows(m, l, h_rows, pos_rows)
    if write_kv:
        K_cache[cache_rows] = k_new
        V_cache[cache_rows] = v_new
    T = K_cache.shape[0]
    o = causal_attention(q, pos_rows, K_cache.reshape(T, Hkv, hd),
                         V_cache.reshape(T, Hkv, hd), Hq, Hkv)
    h1 = h_rows + o.reshape(n, Hq * hd) @ L["w_o"].T
    x2 = rms_norm(h1, L["norm2"], m.norm_eps)
    g = silu(x2 @ L["w_gate"].T) * (x2 @ L["w_up"].T)
    h2 = h1 + g @ L["w_down"].T
    return h2, k_new, v_new


def first_token(m: Model, h_last: np.ndarray) -> int:
    """argmax over the vocabulary of RMSNorm(h_last) E^T (LM head tied to
    the embedding); the first generated token that ends TTFT (QCFuse
    §4.1.5).  Ties resolve to the lowest id."""
    logits = first_token_logits(m, h_last)
    return int(np.argmax(logits))


def first_token_logits(m: Model, h_last: np.ndarray) -> np.ndarray:
    """RMSNorm(h_last) E^T in float64 (the embedding is widened in blocks of
    rows; each logit is still one plain dot product)."""
    x = rms_norm(h_last[None, :], m.final_norm, m.norm_eps)[0]
    out = np.empty(m.embed.shape[0])
    for a in range(0, m.embed.shape[0], 8192):
        out[a:a + 8192] = np.asarray(m.embed[a:a + 8192], dtype=np.float64) @ x
    return out


# --------------------------------------------------------------------------
# full prefill and standalone chunk prefill
# --------------------------------------------------------------------------
@dataclass
class PrefillResult:
    K: np.ndarray          # [n_layers][T][Hkv*hd]
    V: np.ndarray
    hidden: np.ndarray     # [T][d] final hidden states (before final norm)
    token: int             # argmax of the last row's logits


def full_prefill(m: Model, tokens) -> PrefillResult:
    """KV^Full(C) (QCFuse Eq. 2): every token computed under the full
    request at positions 0..T-1, causal attention."""
    tokens = np.asarray(tokens)
    T = len(tokens)
    kvw = m.n_kv_heads * m.head_dim
    K = np.zeros((m.n_layers, T, kvw))
    V = np.zeros((m.n_layers, T, kvw))
    h = embed_rows(m, tokens)
    rows = np.arange(T)
    for l in range(m.n_layers):
        h, _, _ = decoder_layer(m, l, h, rows, K[l], V[l], rows)
    return PrefillResult(K, V, h, first_token(m, h[-1]))


def chunk_prefill(m: Model, chunk_tokens):
    """KV_c^PIC <- LLM(c) (QCFuse Eq. 3): the chunk alone at chunk-local
    positions 0..|c|-1.  Returns (K, V) [n_layers][|c|][Hkv*hd]."""
    r = full_prefill(m, chunk_tokens)
    return r.K, r.V


def chunk_prefill_all(m: Model, chunks):
    """chunk_prefill of every chunk in ``chunks`` (token lists), with the
    layer loop outside the chunk loop: each chunk still runs alone at its
    local positions, through the same decoder_layer calls in the same order
    per chunk, so the result is the per-chunk one bit for bit.  A model
    whose layers are fetched on demand then reads each layer once."""
    kvw = m.n_kv_heads * m.head_dim
    toks = [np.asarray(c) for c in chunks]
    K = [np.zeros((m.n_layers, len(t), kvw)) for t in toks]
    V = [np.zeros((m.n_layers, len(t), kvw)) for t in toks]
    h = [embed_rows(m, t) for t in toks]
    for l in range(m.n_layers):
        for i, t in enumerate(toks):
            rows = np.arange(len(t))
            h[i], _, _ = decoder_layer(m, l, h[i], rows, K[i][l], V[i][l], rows)
    return list(zip(K, V))


# --------------------------------------------------------------------------
# deviation and selection
# --------------------------------------------------------------------------
def kv_deviation(k_current: np.ndarray, k_cached: np.ndarray) -> np.ndarray:
    """d_i = || K_i^current - K_i^cached ||_2^2 over all kv heads and head
    dims ("Request Order Matters" §2.2 Eq. 1).  Rows are tokens."""
    diff = k_current - k_cached
    return np.sum(diff * diff, axis=-1)


def select_count(n_ctx: int, ratio_bp: int) -> int:
    """k = max(1, floor(r N)) ("Request Order Matters" §2.2 Eq. 2; QCFuse Eq.
    8 writes floor(rho N)).  r is given in integer basis points so that the
    floor is exact; r = 0 selects nothing (the direct-reuse endpoint)."""
    if ratio_bp <= 0 or n_ctx <= 0:
        return 0
    return max(1, (n_ctx * ratio_bp) // 10000)


def token_topk(d: np.ndarray, k: int) -> np.ndarray:
    """The k tokens with the largest deviation (LMCache's token top-k,
    "Request Order Matters" §2.2; CacheBlend blog select_hkvd).  Ties go to
    the lower index; the result is sorted ascending by position."""
    order = sorted(range(len(d)), key=lambda i: (-d[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def doc_aligned_select(d: np.ndarray, span_offsets, k: int, order=None) -> np.ndarray:
    """Document-aligned recomputation ("Request Order Matters" §2.3).

    Spans S_j = [span_offsets[j], span_offsets[j+1]).  rho_j is the mean
    deviation over S_j (Eq. 3).  Spans are visited by rho_j descending (ties:
    lower j); whole spans are taken while they fit in the remaining budget;
    at the first span that does not fit, the contiguous window of the
    remaining length with the largest total deviation inside that span is
    taken (ties: leftmost) and selection stops.  Exactly k tokens.  Empty
    spans are skipped.  Sums are float64.

    order: optional visiting order (a permutation of the span indices) that
    replaces the ranking by rho_j -- the random-document control of §2.3,
    whose random order is drawn by the caller."""
    offs = list(span_offsets)
    m = len(offs) - 1
    rho = [float(np.sum(d[offs[j]:offs[j + 1]], dtype=np.float64)) / (offs[j + 1] - offs[j])
           if offs[j + 1] > offs[j] else 0.0 for j in range(m)]
    if order is None:
        idx = sorted(range(m), key=lambda j: (-rho[j], j))
    else:
        idx = [int(j) for j in order]
        assert sorted(idx) == list(range(m)), "order must be a permutation of the spans"
    idx = [j for j in idx if offs[j + 1] > offs[j]]
    spans = [(offs[j], offs[j + 1]) for j in range(m)]
    rem = k
    chosen = []
    for j in idx:
        if rem == 0:
            break
        a, b = spans[j]
        if b - a <= rem:
            chosen.extend(range(a, b))
            rem -= b - a
            continue
        best, best_s = None, -math.inf
        for s in range(a, b - rem + 1):
            tot = float(np.sum(d[s:s + rem], dtype=np.float64))
            if tot > best_s:
                best, best_s = s, tot
        chosen.extend(range(best, best + rem))
        rem = 0
        break
    return np.array(sorted(chosen), dtype=np.int64)


def single_window_select(d: np.ndarray, k: int) -> np.ndarray:
    """Single-window control ("Request Order Matters" §2.3): the contiguous
    k-token window of the reusable tokens with the largest total deviation
    (ties: leftmost).  Sums are float64."""
    n = len(d)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    if k >= n:
        return np.arange(n, dtype=np.int64)
    best, best_s = 0, -math.inf
    for t in range(n - k + 1):
        tot = float(np.sum(d[t:t + k], dtype=np.float64))
        if tot > best_s:
            best, best_s = t, tot
    return np.arange(best, best + k, dtype=np.int64)


def fixed_chunk_offsets(n: int, span_len: int, offset: int):
    """Fixed-chunk spans ("Request Order Matters" §2.3, §4.4): equal spans of
    span_len tokens over the reusable prompt, shifted by `offset` so that
    they cross document boundaries; the first span is [0, offset) and the
    last one is cut at n."""
    offs = [0]
    if 0 < offset < n:
        offs.append(offset)
    while offs[-1] < n:
        offs.append(min(n, offs[-1] + span_len))
    return offs


def first_tokens_select(span_offsets, k: int) -> np.ndarray:
    """Chunk-boundary rule of EPIC's LegoLink (as the QCFuse page describes
    it, §2): a fixed number of the first tokens of every chunk.  The budget
    k is shared out evenly over the non-empty chunks, the first k mod m
    chunks taking one more; a chunk shorter than its share gives the rest
    to the following chunks in order.  Exactly min(k, N) tokens."""
    offs = list(span_offsets)
    spans = [(offs[j], offs[j + 1]) for j in range(len(offs) - 1) if offs[j + 1] > offs[j]]
    m = len(spans)
    if m == 0 or k <= 0:
        return np.zeros(0, dtype=np.int64)
    quota = [k // m + (1 if j < k % m else 0) for j in range(m)]
    take = [min(q, b - a) for q, (a, b) in zip(quota, spans)]
    left = k - sum(take)
    for j, (a, b) in enumerate(spans):
        extra = min(left, (b - a) - take[j])
        take[j] += extra
        left -= extra
    chosen = [i for (a, b), t in zip(spans, take) for i in range(a, a + t)]
    return np.array(chosen, dtype=np.int64)


# --------------------------------------------------------------------------
# blended prefill
# --------------------------------------------------------------------------
@dataclass
class BlendResult:
    K: np.ndarray              # fused cache [n_layers][T][Hkv*hd]
    V: np.ndarray
    selected: np.ndarray       # P: selected context positions, ascending
    deviation: np.ndarray      # d over the N context tokens at layer s
    rows: np.ndarray           # rows computed after layer s (P + always-rows)
    hidden: np.ndarray         # final hidden states of ``rows`` [R][d]
    token: int
    selected_per_layer: dict   # layer -> P used at that layer
    deviation_per_layer: dict = field(default_factory=dict)
    # layer of a gradual-filtering step -> {position: deviation} of the rows
    # ranked there


def blend_prefill(m: Model, segments, store, ratio_bp: int,
                  policy: str = "token_topk", sel_layer: int = 1,
                  span_len: int = 0, span_offset: int = 0, span_order=None,
                  forced=None, schedule=None, forced_steps=None) -> BlendResult:
    """Selective KV recomputation over a partially reused cache (QCFuse
    §2.1.3 Eqs. 6-7; CacheBlend blog ``blend_layer``; LMCache flow of
    "Request Order Matters" §2.2).

    segments: list of (tokens, cached) in request order; cached segments form
      the reusable context C (N tokens), uncached ones (the query U, a new
      document) are recomputed at every layer and are not counted in N.
    store:    list, one entry per cached segment, of (K, V) PIC caches
      [n_layers][len][Hkv*hd] computed standalone at position 0 (Eq. 3).
    forced:   if given, the selected context positions P (ascending) are
      taken from it instead of being ranked (the "forced" mode used for bf16
      parity, where ranking near the k-th deviation is precision dependent).
    policy:   "token_topk" (Eq. 2), "doc_aligned" (Eq. 3), or the §2.3 / §4.4
      controls "single_window", "fixed_chunk" (span_len tokens shifted by
      span_offset; span_len 0 means the median document length shifted by
      half a span),
      "random_doc" (document spans in the order span_order), and
      "first_tokens" (EPIC's chunk-boundary rule).
    schedule: optional gradual filtering (CacheBlend blog select_hkvd):
      list of (layer, keep_count) with layer > sel_layer; at that layer the
      current P is re-ranked by the deviation of its fresh keys and only
      keep_count rows are kept from then on.
    forced_steps: optional {layer: positions} for schedule layers: the
      context positions kept at that step (a subset of the current P, of
      min(keep_count, |P|) entries) are taken from it instead of the
      re-ranking -- the per-step counterpart of ``forced``; the step's
      deviations are still computed.

    Steps:
      1. positions 0..T-1; context positions of cached segments are the
         context token indices 0..N-1 in order (uncached rows interleave at
         their own positions but are not in C).
      2. KV^PIC(C): stitch the store with Pi_i (Eq. 4).
      3. layers < s: full layer on every row (fused = fresh).
      4. layer s: keys of every row are projected fresh; d over context
         tokens (Eq. 1); P = top-k (Eq. 2) or document-aligned spans (Eq. 3).
      5. layers >= s: only P and the uncached rows are computed; their fresh
         K/V replace the PIC entries (Eq. 7) and they attend causally over the
         fused cache; all other rows keep KV^PIC.
      6. first token from the last row.
    """
    Hkv, hd = m.n_kv_heads, m.head_dim
    kvw = Hkv * hd
    toks = np.concatenate([np.asarray(t) for t, _ in segments])
    T = len(toks)
    cached_rows, uncached_rows, lens = [], [], []
    off = 0
    for t, c in segments:
        r = np.arange(off, off + len(t))
        (cached_rows if c else uncached_rows).append(r)
        if c:
            lens.append(len(t))
        off += len(t)
    ctx_rows = np.concatenate(cached_rows) if cached_rows else np.zeros(0, int)
    always = np.concatenate(uncached_rows) if uncached_rows else np.zeros(0, int)
    N = len(ctx_rows)

    # 2. stitched reused cache, placed at the request rows of each chunk.
    # Each chunk is re-rotated by its own request offset.
    K = np.zeros((m.n_layers, T, kvw))
    V = np.zeros((m.n_layers, T, kvw))
    off = 0
    si = 0
    for t, c in segments:
        if c:
            kc, vc = store[si]
            si += 1
            for l in range(m.n_layers):
                K[l, off:off + len(t)] = reposition_keys(kc[l], off, Hkv, hd,
                                                         m.rope_base)
                V[l, off:off + len(t)] = vc[l]
        off += len(t)

    pos_all = np.arange(T)
    h = embed_rows(m, toks)
    # 3. full layers before the selection layer
    for l in range(min(sel_layer, m.n_layers)):
        h, _, _ = decoder_layer(m, l, h, pos_all, K[l], V[l], pos_all)

    k = select_count(N, ratio_bp)
    d = np.zeros(N)
    per_layer = {}
    if sel_layer >= m.n_layers:
        P = np.arange(N)
        active = pos_all
    else:
        # 4. fresh keys of all rows at layer s, deviation over context rows
        L = m.layers[sel_layer]
        x = rms_norm(h, L["norm1"], m.norm_eps)
        qd = m.n_q_heads * hd
        k_all = (x @ L["w_qkv"][qd:qd + kvw].T).reshape(T, Hkv, hd)
        k_all = rope_rotate(k_all, pos_all, m.rope_base).reshape(T, kvw)
        d = kv_deviation(k_all[ctx_rows], K[sel_layer][ctx_rows])
        if forced is not None:
            P = np.asarray(forced, dtype=np.int64)
        elif policy == "token_topk":
            P = token_topk(d, k)
        elif policy == "doc_aligned":
            offs = np.concatenate([[0], np.cumsum(lens)])
            P = doc_aligned_select(d, offs, k)
        elif policy == "random_doc":
            offs = np.concatenate([[0], np.cumsum(lens)])
            P = doc_aligned_select(d, offs, k, order=span_order)
        elif policy == "single_window":
            P = single_window_select(d, k)
        elif policy == "fixed_chunk":
            # span_len 0: the median document length, shifted by half a span
            L_ = span_len if span_len > 0 else max(1, int(np.median(lens)))
            o_ = span_offset if span_len > 0 else L_ // 2
            P = doc_aligned_select(d, fixed_chunk_offsets(N, L_, o_), k)
        elif policy == "first_tokens":
            offs = np.concatenate([[0], np.cumsum(lens)])
            P = first_tokens_select(offs, k)
        else:
            raise ValueError(policy)
        sched = dict(schedule or [])
        dev_steps = {}
        h_act = None
        active = None
        for l in range(sel_layer, m.n_layers):
            if l in sched and l > sel_layer:
                # gradual filtering: re-rank the current P by its fresh keys
                Lw = m.layers[l]
                rows_p = ctx_rows[P]
                sub = np.searchsorted(active, rows_p)
                xp = rms_norm(h_act[sub], Lw["norm1"], m.norm_eps)
                kp = (xp @ Lw["w_qkv"][qd:qd + kvw].T).reshape(-1, Hkv, hd)
                kp = rope_rotate(kp, rows_p, m.rope_base).reshape(-1, kvw)
                dp = kv_deviation(kp, K[l][rows_p])
                dev_steps[l] = dict(zip(P.tolist(), dp.tolist()))
                if forced_steps is not None and l in forced_steps:
                    kept = np.asarray(forced_steps[l], dtype=np.int64)
                    assert len(kept) == min(sched[l], len(P)), "forced step has the wrong size"
                    assert np.all(np.isin(kept, P)), "forced step keeps a row not in P"
                    P = np.sort(kept)
                else:
                    keep = token_topk(dp, min(sched[l], len(P)))
                    P = P[keep]
            new_active = np.union1d(ctx_rows[P], always).astype(np.int64)
            if active is None:
                h_act = h[new_active]
            else:
                h_act = h_act[np.searchsorted(active, new_active)]
            active = new_active
            per_layer[l] = P.copy()
            # 5. Eq. 7 write of fresh K/V, then attention over the fused cache
            h_act, _, _ = decoder_layer(m, l, h_act, active, K[l], V[l], active)
        h_final_rows = active
        tok = first_token(m, h_act[-1])
        return BlendResult(K, V, P, d, h_final_rows, h_act, tok, per_layer, dev_steps)
    tok = first_token(m, h[-1])
    return BlendResult(K, V, P, d, active, h, tok, per_layer)


# --------------------------------------------------------------------------
# byte model
# --------------------------------------------------------------------------
def selection_segments(P) -> int:
    """Number of separate contiguous regions a selection occupies: maximal
    runs of consecutive positions in the ascending set P ("Request Order
    Matters" §4.4, Table 2, "segments")."""
    P = [int(i) for i in P]
    return sum(1 for j, i in enumerate(P) if j == 0 or i != P[j - 1] + 1)


def captured_deviation(P, d) -> float:
    """Share of the selection-layer deviation carried by the selected tokens:
    sum of d_i over P divided by the sum over all reusable tokens ("Request
    Order Matters" §4.4, Table 2, "captured deviation")."""
    d = np.asarray(d, dtype=np.float64)
    total = float(d.sum())
    return float(d[np.asarray(P, dtype=np.int64)].sum()) / total if total > 0 else 0.0


def write_back(result: "BlendResult", segments, m: Model):
    """Cache write-back ("Request Order Matters" §4.2 and §5: each call both
    consumes and updates the persistent cache): after a blended prefill,
    every cached segment's fused K/V rows -- fresh where recomputed, reused
    elsewhere -- are moved back to chunk-local positions (keys rotated by
    minus the segment's request offset, QCFuse Eq. 4 inverted) and become
    that chunk's stored caches.  Returns the new (K, V) [n_layers][len][kvw]
    of each cached segment, in request order."""
    out = []
    off = 0
    for toks, cached in segments:
        n = len(toks)
        if cached:
            K = np.stack([reposition_keys(result.K[l, off:off + n], -off, m.n_kv_heads,
                                          m.head_dim, m.rope_base)
                          for l in range(m.n_layers)])
            V = result.V[:, off:off + n].copy()
            out.append((K, V))
        off += n
    return out


def kv_bytes_per_layer(context_len: int, kv_heads: int, head_dim: int,
                       bytes_per_elem: int = 2) -> int:
    """K plus V bytes of one layer's cache: 2 * L * kv_heads * hd * 2 for
    fp16 (CacheBlend blog, "Hiding Recompute Behind I/O")."""
    return 2 * context_len * kv_heads * head_dim * bytes_per_elem
