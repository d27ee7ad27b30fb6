"""Query-aware selection of QCFuse (§3.2-3.4) in plain float64.

TEST INFRASTRUCTURE ONLY, under the same rules as ``cacheblend.py``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import
it; it shares no code with the CUDA path.

Source: *QCFuse: Query-Aware Cache Fusion via Compressed View for Efficient
RAG Serving* -- §3.2.1 Eqs. 9-11 (full-view selection), §3.3.1 Eq. 14
(per-chunk anchors), §3.3.2 Eqs. 15-17 (anchor-conditioned query probe),
§3.4.2 Eq. 20 (critical-layer score).

Readings taken where the page is silent (each pinned in
``tests/test_oracle_qcfuse.py``):
* Knorm anchors (Eq. 14, "the norm of their key-cache tensors"): the score of
  a chunk-local position is minus the squared L2 norm of its PIC keys summed
  over all layers and kv heads, so the lowest-norm keys rank first (the rule
  of the cited key-norm compression work: low key norm goes with high
  attention).  Sink anchors: the earliest positions of the chunk first.
* anchor count ceil(r_a |c_i|) with r_a in basis points, integer arithmetic;
  ties in any ranking go to the lower position; anchors ascending.
* the query U is every uncached row of the request (they follow the whole
  context); its position ids are its request positions (after C), the
  anchors keep theirs (Eq. 15 and the paragraph after Eq. 17).
* Attn^l(Q, K_C)_t: for every query row and q head, the softmax of
  q.k / sqrt(hd) over the N context keys only, summed over query rows and q
  heads (q head h reads kv head floor(h / (Hq/Hkv))).
* the selection P = TopK(I, k) with k = floor(rho N) as for token top-k
  (Eq. 11; ``select_count``); with P known before any layer runs, the
  blended prefill then recomputes P and U at every layer (selection layer 0).
"""
from __future__ import annotations

import math

import numpy as np

from .cacheblend import (Model, causal_attention, embed_rows, qkv_rows,
                         reposition_keys, rms_norm, select_count, silu,
                         token_topk, blend_prefill)

__all__ = [
    "sink_anchor_scores", "knorm_anchor_scores", "anchor_count", "anchor_positions",
    "probe_query_states", "attention_mass", "query_probe_scores", "query_probe_select",
    "query_probe_blend",
]


# --------------------------------------------------------------------------
# per-chunk anchors (§3.3.1)
# --------------------------------------------------------------------------
def sink_anchor_scores(n: int) -> np.ndarray:
    """G_i(r) of the Sink rule: the earliest chunk positions rank highest."""
    return -np.arange(n, dtype=np.float64)


def knorm_anchor_scores(k_chunk: np.ndarray) -> np.ndarray:
    """G_i(r) of the Knorm rule for one chunk's PIC keys k_chunk
    [n_layers][n][Hkv*hd]: minus the squared L2 norm of the position's keys
    summed over layers and kv heads (lowest norm ranks first)."""
    return -np.sum(k_chunk * k_chunk, axis=(0, 2))


def anchor_count(n: int, ratio_bp: int) -> int:
    """ceil(r_a |c_i|) of Eq. 14 with r_a = ratio_bp / 10000."""
    return (n * ratio_bp + 9999) // 10000


def anchor_positions(scores: np.ndarray, ratio_bp: int) -> np.ndarray:
    """A_i = TopK(G_i, ceil(r_a |c_i|)) (Eq. 14), chunk-local, ascending."""
    return token_topk(np.asarray(scores, dtype=np.float64), anchor_count(len(scores), ratio_bp))


# --------------------------------------------------------------------------
# anchor-conditioned query probe (§3.3.2; §3.2.1 when every position is kept)
# --------------------------------------------------------------------------
def probe_query_states(m: Model, u_tokens, u_pos, K_pre, V_pre, last_layer: int):
    """Q_U^l(C_A) <- LLM^l(U; KV^A(C_A)) (Eq. 17; Eq. 9 with the whole
    context as prefix).

    u_tokens, u_pos: the query rows and their request positions.  K_pre,
    V_pre [n_layers][n_pre][Hkv*hd]: the prefix cache rows (stitched PIC
    entries at their request positions, all before u_pos), read only.  The
    query rows run layers 0..last_layer over [prefix; U]: row i sees every
    prefix row and query rows 0..i.  Returns {l: (q, k)} with the query rows'
    post-RoPE q [n_u, Hq, hd] and fresh k [n_u, Hkv*hd] entering layer l."""
    Hq, Hkv, hd = m.n_q_heads, m.n_kv_heads, m.head_dim
    h = embed_rows(m, u_tokens)
    n_u = h.shape[0]
    n_pre = K_pre.shape[1]
    out = {}
    for l in range(last_layer + 1):
        q, k, v = qkv_rows(m, l, h, u_pos)
        out[l] = (q, k)
        if l == last_layer:
            break
        K = np.concatenate([K_pre[l], k], 0).reshape(n_pre + n_u, Hkv, hd)
        V = np.concatenate([V_pre[l], v], 0).reshape(n_pre + n_u, Hkv, hd)
        o = causal_attention(q, n_pre + np.arange(n_u), K, V, Hq, Hkv)
        L = m.layers[l]
        h = h + o.reshape(n_u, Hq * hd) @ L["w_o"].T
        x2 = rms_norm(h, L["norm2"], m.norm_eps)
        h = h + (silu(x2 @ L["w_gate"].T) * (x2 @ L["w_up"].T)) @ L["w_down"].T
    return out


def attention_mass(q: np.ndarray, K_ctx: np.ndarray, n_q_heads: int, n_kv_heads: int):
    """Attn(Q_U, K_C)_t of §3.2.1: the user-query-to-context attention mass on
    context position t.  q [n_u, Hq, hd]; K_ctx [N, Hkv*hd].  For each query
    row and q head, softmax(q.k / sqrt(hd)) over the N context keys; the
    probabilities are summed over rows and heads.  Returns [N]."""
    n_u, Hq, hd = q.shape
    N = K_ctx.shape[0]
    group = n_q_heads // n_kv_heads
    K = K_ctx.reshape(N, n_kv_heads, hd)
    mass = np.zeros(N)
    for h in range(Hq):
        s = (q[:, h, :] @ K[:, h // group, :].T) / math.sqrt(hd)   # [n_u, N]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        mass += p.sum(axis=0)
    return mass


def query_probe_scores(m: Model, u_tokens, u_pos, K_ctx, V_ctx, anchors, crit_layers):
    """I_{L*}(t) = sum_{l in L*} Attn^l(Q_U^l(C_A), K_C^{PIC,l})_t (Eq. 20).

    K_ctx, V_ctx [n_layers][N][Hkv*hd]: the stitched KV^PIC(C) (Eq. 4).
    anchors: ascending context positions of C_A (Eqs. 15-16).  With every
    position an anchor and L* every layer this is the full-view score of
    Eq. 10."""
    last = max(crit_layers)
    qs = probe_query_states(m, u_tokens, u_pos, K_ctx[:, anchors], V_ctx[:, anchors], last)
    N = K_ctx.shape[1]
    I = np.zeros(N)
    for l in sorted(set(crit_layers)):
        I += attention_mass(qs[l][0], K_ctx[l], m.n_q_heads, m.n_kv_heads)
    return I


def query_probe_select(m: Model, segments, store, ratio_bp: int, anchor_rule: str = "knorm",
                       anchor_bp: int = 1000, crit_layers=None):
    """P(U, C) = TopK(I(t), floor(rho N)) (Eq. 11) with I from Eq. 20.

    segments / store as for ``blend_prefill`` (cached segments first, then
    the uncached rows U).  anchor_rule: "sink" or "knorm" per chunk
    (Eq. 14, ratio anchor_bp), or "all" (every position: the full view,
    Eq. 9).  crit_layers: the critical-layer set L* (None: every layer,
    Eq. 10).  Returns (P, I, anchors) with anchors as context positions."""
    Hkv, hd = m.n_kv_heads, m.head_dim
    cached = [(np.asarray(t), i) for i, (t, c) in enumerate(segments) if c]
    u_tokens = np.concatenate([np.asarray(t) for t, c in segments if not c])
    # stitched KV^PIC(C) of the context positions (Eq. 4)
    Ks, Vs, anchors = [], [], []
    off = 0
    for si, (t, _) in enumerate(cached):
        kc, vc = store[si]
        n = len(t)
        Ks.append(np.stack([reposition_keys(kc[l], off, Hkv, hd, m.rope_base)
                            for l in range(m.n_layers)]))
        Vs.append(np.asarray(vc, dtype=np.float64))
        if anchor_rule == "all":
            a = np.arange(n)
        elif anchor_rule == "sink":
            a = anchor_positions(sink_anchor_scores(n), anchor_bp)
        elif anchor_rule == "knorm":
            a = anchor_positions(knorm_anchor_scores(np.asarray(kc, dtype=np.float64)), anchor_bp)
        else:
            raise ValueError(anchor_rule)
        anchors.append(a + off)
        off += n
    N = off
    K_ctx = np.concatenate(Ks, 1)
    V_ctx = np.concatenate(Vs, 1)
    anchors = np.concatenate(anchors).astype(np.int64)
    crit = list(range(m.n_layers)) if crit_layers is None else list(crit_layers)
    u_pos = N + np.arange(len(u_tokens))
    I = query_probe_scores(m, u_tokens, u_pos, K_ctx, V_ctx, anchors, crit)
    P = token_topk(I, select_count(N, ratio_bp))
    return P, I, anchors


def query_probe_blend(m: Model, segments, store, ratio_bp: int, anchor_rule: str = "knorm",
                      anchor_bp: int = 1000, crit_layers=None):
    """The selector's P handed to selective recomputation (§3.5): P is known
    before any layer runs, so every layer recomputes P and U over the fused
    cache (QCFuse Eq. 7).  Returns (BlendResult, I, anchors)."""
    P, I, anchors = query_probe_select(m, segments, store, ratio_bp, anchor_rule, anchor_bp,
                                       crit_layers)
    res = blend_prefill(m, segments, store, ratio_bp, sel_layer=0, forced=P)
    return res, I, anchors
