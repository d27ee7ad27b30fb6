"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds shapes, workload recipes and random-number generation only.
It performs none of the method's arithmetic: no RoPE, no attention, no
deviation, no selection.  Both the CPU oracle (``oracle/``) and the CUDA path
(``rag_kv_cache_layer_gb300``) consume what it produces; neither side's
results ever flow back into it.

Recipes (the pages' workloads are LongBench/RULER requests split into
512-token chunks with 20 chunks per request, QCFuse §4.1.4, and an
84-document rolling finance window, "Request Order Matters" §4.1; neither
dataset is available, so seeded synthetic token streams of the same shape
stand in for them):

* weights: every projection matrix N(0, 0.02), embeddings N(0, 1), RMSNorm
  gains 1, no biases; bf16 models round each value to the nearest bf16
  (round-to-nearest-even) so that both sides see identical numbers.
* token ids: uniform over the vocabulary, drawn per chunk / document.
* requests: a list of cached segments (chunks or documents) followed by
  uncached segments (the user query, plus in the rolling workload the newly
  appended document), positions 0..T-1 in that order.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np


# --------------------------------------------------------------------------
# model shapes
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    rope_base: float = 10000.0
    norm_eps: float = 1e-5
    dtype: str = "bf16"          # "f32" or "bf16": storage type of weights / KV

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def kv_row_elems(self) -> int:
        return self.n_kv_heads * self.head_dim

    def truncated(self, n_layers: int) -> "ModelShape":
        return dataclasses.replace(self, n_layers=n_layers,
                                   name=f"{self.name}-{n_layers}L")


TINY_F32 = ModelShape("tiny", 2, 256, 4, 2, 64, 688, 4096, dtype="f32")
LLAMA3_8B = ModelShape("llama3-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256)
# The vocabulary of the Qwen3-8B shape is not given by the workload text; the
# public Qwen3 tokenizer size is used (it only changes the LM-head GEMV).
QWEN3_8B = ModelShape("qwen3-8b-shape", 36, 4096, 32, 8, 128, 12288, 151936)


# --------------------------------------------------------------------------
# request descriptions
# --------------------------------------------------------------------------
@dataclass
class Segment:
    """A run of request tokens.  ``chunk_id`` >= 0 names a cached chunk in the
    store (reusable context); ``chunk_id`` == -1 marks an uncached segment
    that is recomputed at every layer (the user query, a new document)."""
    tokens: np.ndarray          # int32 [len]
    chunk_id: int = -1

    @property
    def cached(self) -> bool:
        return self.chunk_id >= 0


@dataclass
class Request:
    segments: list

    @property
    def tokens(self) -> np.ndarray:
        return np.concatenate([s.tokens for s in self.segments]).astype(np.int32)

    @property
    def n_tokens(self) -> int:
        return int(sum(len(s.tokens) for s in self.segments))

    @property
    def n_ctx(self) -> int:
        return int(sum(len(s.tokens) for s in self.segments if s.cached))


@dataclass
class Workload:
    name: str
    model: ModelShape
    seed: int
    ratio_bp: int                # recompute ratio in basis points
    policy: str                  # "token_topk" | "doc_aligned"
    chunks: list                 # list of int32 token arrays (the chunk pool)
    requests: list               # list[Request]
    sel_layer: int = 1
    extra: dict = field(default_factory=dict)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even) and return
    them as float32 values (exactly representable in bf16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = ((bits + 0x7FFF + lsb) >> 16) << 16
    return bits.astype(np.uint32).view(np.float32)


def _normal(rng, shape, std, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == "bf16":
        x = round_to_bf16(x)
    return x


def make_weights(model: ModelShape, seed: int, std: float = 0.02,
                 embed_std: float = 1.0) -> dict:
    """Random-init decoder weights, float32 arrays holding (for bf16 models)
    bf16-exact values.  Layout: each projection is [out_features, in_features]
    (row n holds the weights of output n).  ``w_qkv`` stacks W_q, W_k, W_v
    along the output dimension."""
    rng = np.random.default_rng(seed)
    d, F = model.d_model, model.d_ffn
    qd = model.n_q_heads * model.head_dim
    w = {
        "embed": _normal(rng, (model.vocab, d), embed_std, model.dtype),
        "final_norm": np.ones(d, np.float32),
        "layers": [],
    }
    for _ in range(model.n_layers):
        w["layers"].append({
            "w_qkv": _normal(rng, (model.qkv_rows, d), std, model.dtype),
            "w_o": _normal(rng, (d, qd), std, model.dtype),
            "w_gate": _normal(rng, (F, d), std, model.dtype),
            "w_up": _normal(rng, (F, d), std, model.dtype),
            "w_down": _normal(rng, (d, F), std, model.dtype),
            "norm1": np.ones(d, np.float32),
            "norm2": np.ones(d, np.float32),
        })
    return w


def make_weights_device(model: ModelShape, seed: int, device, std: float = 0.02,
                        embed_std: float = 1.0) -> dict:
    """Random-init bf16 weights generated on a CUDA device with torch's seeded
    generator (for stacks too large to draw on the host): projections
    N(0, std), embeddings N(0, embed_std), RMSNorm gains 1.  Same layout as
    make_weights, as device tensors."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def rnd(*shape, s=std):
        return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
                * s).to(torch.bfloat16)
    d, F = model.d_model, model.d_ffn
    qd = model.n_q_heads * model.head_dim
    w = {"embed": rnd(model.vocab, d, s=embed_std),
         "final_norm": torch.ones(d, device=device), "layers": []}
    for _ in range(model.n_layers):
        w["layers"].append({
            "w_qkv": rnd(model.qkv_rows, d), "w_o": rnd(d, qd),
            "w_gate": rnd(F, d), "w_up": rnd(F, d), "w_down": rnd(d, F),
            "norm1": torch.ones(d, device=device), "norm2": torch.ones(d, device=device)})
    return w


def make_tokens(rng, n, vocab) -> np.ndarray:
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def make_kv_store(model: ModelShape, n_rows: int, seed: int, std: float = 1.0):
    """Synthetic per-layer K and V rows [n_layers][n_rows][Hkv*hd] (used by
    kernel-level tests and timing samples where the values need not come
    from a chunk prefill)."""
    rng = np.random.default_rng(seed)
    shape = (model.n_layers, n_rows, model.kv_row_elems)
    return (_normal(rng, shape, std, model.dtype),
            _normal(rng, shape, std, model.dtype))


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
def tiny_blend(seed: int = 0, n_chunks: int = 3, chunk_len: int = 128,
               n_query: int = 32, ratio_bp: int = 1500,
               n_layers: int | None = None) -> Workload:
    """2-layer fp32 model (deeper with n_layers); 3 chunks x 128 tokens + 32
    query tokens; 15%."""
    rng = np.random.default_rng(seed + 1000)
    m = TINY_F32 if n_layers is None else TINY_F32.truncated(n_layers)
    chunks = [make_tokens(rng, chunk_len, m.vocab) for _ in range(n_chunks)]
    segs = [Segment(c, i) for i, c in enumerate(chunks)]
    segs.append(Segment(make_tokens(rng, n_query, m.vocab)))
    return Workload("tiny_fp32", m, seed, ratio_bp, "token_topk", chunks,
                    [Request(segs)])


def llama_rag(seed: int = 1, n_layers: int | None = None, n_chunks: int = 6,
              chunk_len: int = 512, n_query: int = 64,
              ratio_bp: int = 1500) -> Workload:
    """Llama-3-8B-shaped stack; 6 chunks x 512 + 64 query tokens; 15%; B=1."""
    m = LLAMA3_8B if n_layers is None else LLAMA3_8B.truncated(n_layers)
    rng = np.random.default_rng(seed + 1000)
    chunks = [make_tokens(rng, chunk_len, m.vocab) for _ in range(n_chunks)]
    segs = [Segment(c, i) for i, c in enumerate(chunks)]
    segs.append(Segment(make_tokens(rng, n_query, m.vocab)))
    return Workload("llama8b_rag_6x512_ratio15pct", m, seed, ratio_bp, "token_topk",
                    chunks, [Request(segs)])


def qwen_pool(seed: int = 2, n_layers: int | None = None, pool: int = 40,
              per_req: int = 10, chunk_len: int = 1024, n_query: int = 128,
              batch: int = 4, ratio_bp: int = 3000) -> Workload:
    """Qwen3-8B-shaped stack; each of 4 requests draws 10 of a 40-chunk pool
    in a seeded random order, + 128 query tokens; 30%."""
    m = QWEN3_8B if n_layers is None else QWEN3_8B.truncated(n_layers)
    rng = np.random.default_rng(seed + 1000)
    chunks = [make_tokens(rng, chunk_len, m.vocab) for _ in range(pool)]
    reqs = []
    for _ in range(batch):
        order = rng.choice(pool, size=per_req, replace=False)
        segs = [Segment(chunks[i], int(i)) for i in order]
        segs.append(Segment(make_tokens(rng, n_query, m.vocab)))
        reqs.append(Request(segs))
    return Workload("qwen8b_pool40_10x1024_b4_ratio30pct", m, seed, ratio_bp,
                    "token_topk", chunks, reqs)


def long_context(seed: int = 3, n_layers: int | None = None,
                 n_chunks: int = 32, chunk_len: int = 1024,
                 n_query: int = 256, batch: int = 2,
                 ratio_bp: int = 500) -> Workload:
    """Llama shape; 32 chunks x 1024 (32K context) + 256 query; B=2."""
    m = LLAMA3_8B if n_layers is None else LLAMA3_8B.truncated(n_layers)
    rng = np.random.default_rng(seed + 1000)
    chunks, reqs = [], []
    for _ in range(batch):
        segs = []
        for _ in range(n_chunks):
            chunks.append(make_tokens(rng, chunk_len, m.vocab))
            segs.append(Segment(chunks[-1], len(chunks) - 1))
        segs.append(Segment(make_tokens(rng, n_query, m.vocab)))
        reqs.append(Request(segs))
    return Workload(f"llama8b_long32k_b2_r{ratio_bp // 100}", m, seed,
                    ratio_bp, "token_topk", chunks, reqs)


def rolling_stream(seed: int = 4, n_layers: int | None = None,
                   window: int = 20, doc_len: int = 400, n_query: int = 64,
                   n_requests: int = 50, ratio_bp: int = 500,
                   policy: str = "doc_aligned") -> Workload:
    """Rolling-agent window: a stream of seeded 400-token documents; request t
    holds documents t..t+window-1 followed by a query.  The newest document
    has no cache when request t is evaluated (the previous window's
    documents are populated first), so it is an uncached segment; every other
    document is a cached chunk whose store persists across requests."""
    m = LLAMA3_8B if n_layers is None else LLAMA3_8B.truncated(n_layers)
    rng = np.random.default_rng(seed + 1000)
    n_docs = window + n_requests - 1
    docs = [make_tokens(rng, doc_len, m.vocab) for _ in range(n_docs)]
    reqs = []
    for t in range(n_requests):
        segs = [Segment(docs[i], i) for i in range(t, t + window - 1)]
        segs.append(Segment(docs[t + window - 1]))        # newly appended
        segs.append(Segment(make_tokens(rng, n_query, m.vocab)))
        reqs.append(Request(segs))
    return Workload(f"llama8b_rolling_{window}x{doc_len}_{policy}", m, seed,
                    ratio_bp, policy, docs, reqs)
