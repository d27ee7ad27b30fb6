"""Edge shapes through the whole blended prefill against the oracle:

* ragged chunks (1, 37, 200 and 63 tokens) and a 5-token query on the fp32
  model, so no length is a multiple of a tile, a block or a warp;
* the largest batch one call takes (CB_MAX_BATCH = 64 requests of two short
  chunks and a 1-4-token query each, drawn from a shared pool), each
  request checked alone against the oracle;
* the degenerate budgets: one cached token with the smallest nonzero ratio
  (k = max(1, floor(N r)) = 1, the only token) and r = 0 (pure reuse), with
  a one-token query; a request with no cached chunk (N = 0) in a batch;
* the bf16 tensor-core path on ragged chunks (100, 333 and 7 tokens + 13
  query tokens) with the oracle's selection imposed: row counts that leave
  partial GEMM tiles and attention tiles everywhere.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L
from gpu_common import assert_close, host, rms_rel, ties_ok

pytestmark = pytest.mark.gpu


class Stack:
    """A model on the device and in the oracle, with a chunk pool in both."""

    def __init__(self, shape, seed, chunks, max_pos=4096):
        self.shape = shape
        self.weights = W.make_weights(shape, seed)
        self.model = R.BlendModel.from_host(shape, self.weights, max_pos)
        self.om = O.model_from_weights(shape, self.weights)
        self.chunks = chunks
        self.store = R.ChunkStore(self.model, sum(len(c) for c in chunks))
        self.store.prefill({i: torch.from_numpy(c).cuda() for i, c in enumerate(chunks)})
        self.ostore = O.chunk_prefill_all(self.om, chunks)
        torch.cuda.synchronize()

    def gpu_req(self, chunk_ids, query):
        toks = np.concatenate([self.chunks[i] for i in chunk_ids] + [query]).astype(np.int32)
        segs = [self.store.seg(i) for i in chunk_ids] + [R.Seg(len(query))]
        return R.Req(torch.from_numpy(toks).cuda(), segs)

    def oracle(self, chunk_ids, query, ratio_bp, **kw):
        segs = [(self.chunks[i], True) for i in chunk_ids] + [(query, False)]
        return O.blend_prefill(self.om, segs, [self.ostore[i] for i in chunk_ids], ratio_bp, **kw)


def _check_fp32(out, ref, t0, T, r0, k0, k):
    """Request at fused-cache rows [t0, t0 + T), computed rows from r0,
    selection from k0."""
    sel = out["selected"][k0:k0 + k].cpu().numpy()
    assert ties_ok(sel, ref.selected, ref.deviation, k)
    if set(sel.tolist()) == set(ref.selected.tolist()):
        assert_close(host(out["k_cache"][:, t0:t0 + T]), ref.K, torch.float32)
        assert_close(host(out["v_cache"][:, t0:t0 + T]), ref.V, torch.float32)
        Rn = len(ref.rows)
        assert np.array_equal(out["rows"][r0:r0 + Rn].cpu().numpy(), ref.rows)
        assert_close(host(out["hidden"][r0:r0 + Rn]), ref.hidden, torch.float32)


def test_ragged_chunks_fp32():
    rng = np.random.default_rng(5)
    shape = W.TINY_F32
    chunks = [W.make_tokens(rng, n, shape.vocab) for n in (1, 37, 200, 63)]
    st = Stack(shape, 3, chunks)
    query = W.make_tokens(rng, 5, shape.vocab)
    ids = [0, 1, 2, 3]
    out = st.model.cb_blend_prefill([st.gpu_req(ids, query)], 1500)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    ref = st.oracle(ids, query, 1500)
    assert len(ref.selected) == O.select_count(301, 1500) == 45
    _check_fp32(out, ref, 0, 306, 0, 0, 45)


def test_largest_batch_fp32():
    rng = np.random.default_rng(6)
    shape = W.TINY_F32
    pool = [W.make_tokens(rng, int(rng.integers(1, 25)), shape.vocab) for _ in range(40)]
    st = Stack(shape, 4, pool)
    B = L.CB_MAX_BATCH
    picks = [rng.choice(len(pool), size=2, replace=False).tolist() for _ in range(B)]
    queries = [W.make_tokens(rng, int(rng.integers(1, 5)), shape.vocab) for _ in range(B)]
    reqs = [st.gpu_req(p, q) for p, q in zip(picks, queries)]
    out = st.model.cb_blend_prefill(reqs, 3000)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    t0 = r0 = k0 = 0
    for p, q in zip(picks, queries):
        ref = st.oracle(p, q, 3000)
        T = sum(len(pool[i]) for i in p) + len(q)
        k = len(ref.selected)
        _check_fp32(out, ref, t0, T, r0, k0, k)
        t0, r0, k0 = t0 + T, r0 + len(ref.rows), k0 + k
    with pytest.raises(L.CBError):          # one more request than a call takes
        st.model.cb_blend_prefill(reqs + reqs[:1], 3000)


@pytest.mark.parametrize("ratio_bp", [1, 0])
def test_one_cached_token_budgets(ratio_bp):
    rng = np.random.default_rng(7)
    shape = W.TINY_F32
    chunks = [W.make_tokens(rng, 1, shape.vocab)]
    st = Stack(shape, 5, chunks)
    query = W.make_tokens(rng, 1, shape.vocab)
    out = st.model.cb_blend_prefill([st.gpu_req([0], query)], ratio_bp)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    ref = st.oracle([0], query, ratio_bp)
    k = O.select_count(1, ratio_bp)
    assert len(ref.selected) == k == (1 if ratio_bp else 0)
    _check_fp32(out, ref, 0, 2, 0, 0, k)
    assert int(out["first_token"][0]) == ref.token or \
        O.first_token_logits(st.om, ref.hidden[-1])[int(out["first_token"][0])] >= \
        O.first_token_logits(st.om, ref.hidden[-1]).max() - 1e-4


def test_request_without_cached_chunks_in_a_batch_fp32():
    """A request whose context has no cached chunk (N = 0, so k = 0: every
    row is computed at every layer) batched after a normal one.  Each
    request against the oracle; the chunk-less one also equals a full
    prefill of its tokens alone (the same sums in the same order)."""
    rng = np.random.default_rng(11)
    shape = W.TINY_F32
    chunks = [W.make_tokens(rng, n, shape.vocab) for n in (64, 96)]
    st = Stack(shape, 13, chunks)
    q0 = W.make_tokens(rng, 9, shape.vocab)
    q1 = W.make_tokens(rng, 41, shape.vocab)
    bare = R.Req(torch.from_numpy(q1.astype(np.int32)).cuda(), [R.Seg(len(q1))])
    out = st.model.cb_blend_prefill([st.gpu_req([0, 1], q0), bare], 1500)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    k0 = O.select_count(160, 1500)
    ref0 = st.oracle([0, 1], q0, 1500)
    _check_fp32(out, ref0, 0, 169, 0, 0, k0)
    ref1 = O.blend_prefill(st.om, [(q1, False)], [], 1500)
    assert len(ref1.selected) == 0 and len(ref1.rows) == 41
    R0 = len(ref0.rows)
    _check_fp32(out, ref1, 169, 41, R0, k0, 0)
    full = st.model.cb_full_prefill([bare])
    torch.cuda.synchronize()
    assert torch.equal(out["k_cache"][:, 169:210], full["k_cache"][:, :41])
    assert torch.equal(out["v_cache"][:, 169:210], full["v_cache"][:, :41])
    assert int(out["first_token"][1]) == int(full["first_token"][0])


def test_ragged_chunks_bf16_forced():
    rng = np.random.default_rng(8)
    shape = W.LLAMA3_8B.truncated(2)
    chunks = [W.make_tokens(rng, n, shape.vocab) for n in (100, 333, 7)]
    st = Stack(shape, 9, chunks)
    query = W.make_tokens(rng, 13, shape.vocab)
    ids = [0, 1, 2]
    ref = st.oracle(ids, query, 1500)
    forced = torch.from_numpy(ref.selected.astype(np.int32)).cuda()
    out = st.model.cb_blend_prefill([st.gpu_req(ids, query)], 1500, forced=forced)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    for l in range(2):
        assert rms_rel(host(out["k_cache"][l]), ref.K[l]) <= 2e-2
        assert rms_rel(host(out["v_cache"][l]), ref.V[l]) <= 2e-2
    Rn = len(ref.rows)
    assert np.array_equal(out["rows"][:Rn].cpu().numpy(), ref.rows)
    assert rms_rel(host(out["hidden"][:Rn]), ref.hidden) <= 2e-2
    # the GPU's own ranking on the same request: exact top-k of its own d
    free = st.model.cb_blend_prefill([st.gpu_req(ids, query)], 1500)
    N, k = 440, len(ref.selected)
    d = free["deviation"][:N].cpu().numpy().astype(np.float64)
    assert list(free["selected"][:k].cpu().numpy()) == list(O.token_topk(d, k))
    assert rms_rel(d, ref.deviation) <= 2e-2


@pytest.fixture
def index_checks():
    L.check(L.lib.cb_debug_index_checks(1))
    yield
    L.check(L.lib.cb_debug_index_checks(0))


def test_index_checks_pass_correct_calls_and_change_nothing(index_checks):
    rng = np.random.default_rng(9)
    shape = W.TINY_F32
    chunks = [W.make_tokens(rng, n, shape.vocab) for n in (50, 70)]
    st = Stack(shape, 6, chunks)
    query = W.make_tokens(rng, 9, shape.vocab)
    on = st.model.cb_blend_prefill([st.gpu_req([0, 1], query)], 2000,
                                   schedule=[(1, 5)] if shape.n_layers > 2 else None)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    L.check(L.lib.cb_debug_index_checks(0))
    off = st.model.cb_blend_prefill([st.gpu_req([0, 1], query)], 2000)
    torch.cuda.synchronize()
    for key in ("k_cache", "v_cache", "selected", "rows", "first_token"):
        assert torch.equal(on[key], off[key]), key


def test_index_checks_report_an_unsorted_forced_selection(index_checks):
    """A forced selection in range but out of order: without the checks the
    call runs (on wrong rows); with them the status word says so."""
    rng = np.random.default_rng(10)
    shape = W.TINY_F32
    chunks = [W.make_tokens(rng, 40, shape.vocab)]
    st = Stack(shape, 7, chunks)
    query = W.make_tokens(rng, 4, shape.vocab)
    k = O.select_count(40, 1000)
    bad = torch.arange(k, 0, -1, dtype=torch.int32, device="cuda")      # descending
    st.model.cb_blend_prefill([st.gpu_req([0], query)], 1000, forced=bad)
    torch.cuda.synchronize()
    assert R.device_status() == L.CB_ERR_DEVICE_INDEX
    assert R.device_status() == 0


def test_index_checks_report_unsorted_attention_positions(index_checks):
    n_q, T = 8, 64
    q = torch.randn(n_q, 4 * 64, device="cuda")
    kc = torch.randn(T, 2 * 64, device="cuda")
    vc = torch.randn(T, 2 * 64, device="cuda")
    out = torch.empty_like(q)
    good = torch.arange(10, 10 + n_q, dtype=torch.int32, device="cuda")
    R.cb_sparse_query_attention(q, good, [(0, n_q, 0, T)], kc, vc, 4, 2, 64, out)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    R.cb_sparse_query_attention(q, good.flip(0), [(0, n_q, 0, T)], kc, vc, 4, 2, 64, out)
    torch.cuda.synchronize()
    assert R.device_status() == L.CB_ERR_DEVICE_INDEX
