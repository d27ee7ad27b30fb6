"""Parity of the query-aware selectors (QCFuse §3.2-3.4) on the CUDA path
against the oracle, on a Llama-3-8B-shaped bf16 stack truncated to 3 layers
(2 chunks x 256 + 64 query tokens):

* anchors (Eq. 14): the GPU's Knorm scores against the oracle's on the same
  PIC keys (float accumulation, 1e-4 relative); the anchors exactly the
  per-chunk top-k of the GPU's own scores; Sink anchors exactly the heads of
  the chunks;
* the score I(t) (Eq. 20, and Eq. 10 for the full view) against the
  oracle's probe of its own float64 chunk caches with the same anchors and
  critical layers, at 5e-2 RMS-relative (a softmax-weighted sum of bf16
  projections); P exactly the top-k of the GPU's own I (Eq. 11);
* the blended prefill that follows against the oracle's blend with the GPU's
  P from layer 0, at 2e-2 RMS-relative, as for the other policies.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L
from gpu_common import host, rms_rel
from test_gpu_blend import Setup, _host_store

pytestmark = pytest.mark.gpu

TOL_I = 5e-2
TOL = 2e-2


@pytest.fixture(scope="module")
def q3():
    return Setup(W.llama_rag(n_layers=3, n_chunks=2, chunk_len=256, n_query=64), max_pos=4096)


def _chunks(st):
    rq = st.wl.requests[0]
    return [s for s in rq.segments if s.cached]


def _oracle_inputs(st):
    rq = st.wl.requests[0]
    segs = [(s.tokens, s.cached) for s in rq.segments]
    store = [st.ostore[s.chunk_id] for s in rq.segments if s.cached]
    return segs, store


def test_knorm_anchor_scores_and_ranking(q3):
    chunks = _chunks(q3)
    segs = [q3.store.seg(s.chunk_id) for s in chunks]
    anchors, scores = q3.model.cb_anchor_select(segs, L.CB_ANCHOR_KNORM, 1000)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    a, sc = anchors.cpu().numpy(), scores.cpu().numpy().astype(np.float64)
    off_s = off_a = 0
    for s in chunks:
        r, n = q3.store.where[s.chunk_id]
        k = host(q3.store.K[:, r:r + n])                      # the GPU's PIC keys
        ref = O.knorm_anchor_scores(k)
        got = sc[off_s:off_s + n]
        assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))
        cnt = O.anchor_count(n, 1000)
        assert list(a[off_a:off_a + cnt]) == list(O.anchor_positions(got, 1000))
        off_s += n
        off_a += cnt


def test_sink_anchors_are_chunk_heads(q3):
    segs = [q3.store.seg(s.chunk_id) for s in _chunks(q3)]
    anchors, scores = q3.model.cb_anchor_select(segs, L.CB_ANCHOR_SINK, 2500)
    torch.cuda.synchronize()
    want = [i for s in segs for i in range(O.anchor_count(s.len, 2500))]
    assert list(anchors.cpu().numpy()) == want


@pytest.mark.parametrize("policy,query,rule,bp,crit", [
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_SINK, "anchor_bp": 1000,
                               "crit_layers": [1, 2]}, "sink", 1000, [1, 2]),
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_SINK, "anchor_bp": 2500,
                               "crit_layers": [0]}, "sink", 2500, [0]),
    (L.CB_POLICY_QUERY_FULL, None, "all", 0, None),
])
def test_query_probe_blend(q3, policy, query, rule, bp, crit):
    N = sum(s.len for s in [q3.store.seg(c.chunk_id) for c in _chunks(q3)])
    out = q3.model.cb_blend_prefill(q3.gpu_reqs(), 1500, policy=policy, sel_layer=0,
                                    query=query)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    I_gpu = out["deviation"][:N].cpu().numpy().astype(np.float64)
    k = O.select_count(N, 1500)
    P_gpu = out["selected"][:k].cpu().numpy()
    # Eq. 11 on the GPU's own scores, exactly
    assert list(P_gpu) == list(O.token_topk(I_gpu, k))
    # Eq. 20 / Eq. 10 against the oracle
    segs, store = _oracle_inputs(q3)
    P_ref, I_ref, _ = O.query_probe_select(q3.om, segs, store, 1500, rule, bp, crit)
    n_crit = q3.shape.n_layers if crit is None else len(crit)
    assert abs(I_gpu.sum() - n_crit * 64 * q3.shape.n_q_heads) <= 1e-3 * I_gpu.sum()
    assert rms_rel(I_gpu, I_ref) <= TOL_I
    # the blend with the GPU's P from layer 0
    ref = O.blend_prefill(q3.om, segs, store, 1500, sel_layer=0, forced=P_gpu)
    for l in range(q3.shape.n_layers):
        assert rms_rel(host(out["k_cache"][l]), ref.K[l]) <= TOL
        assert rms_rel(host(out["v_cache"][l]), ref.V[l]) <= TOL
    Rn = len(ref.rows)
    assert rms_rel(host(out["hidden"][:Rn]), ref.hidden) <= TOL


@pytest.mark.parametrize("ctas", [0, 2], ids=["copy_engines", "zero_copy_2_ctas"])
@pytest.mark.parametrize("policy,query,rule,bp,crit", [
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_SINK, "anchor_bp": 1000,
                               "crit_layers": [1, 2]}, "sink", 1000, [1, 2]),
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_KNORM, "anchor_bp": 1000,
                               "crit_layers": [0, 1]}, None, 1000, [0, 1]),
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_KNORM, "anchor_bp": 1000,
                               "crit_layers": [1, 2], "anchors": "given"}, None, 1000, [1, 2]),
    (L.CB_POLICY_QUERY_FULL, None, "all", 0, None),
], ids=["probe_sink", "probe_knorm", "probe_given_anchors", "full_view"])
def test_query_policies_on_host_resident_chunks(q3, policy, query, rule, bp, crit, ctas):
    """[CB] "Hiding Recompute Behind I/O" with QCFuse's selectors: the chunk
    caches stay in pinned host memory and arrive layer by layer (the layers
    the probe reads first; Knorm scores read the host keys in a kernel).
    Against the device-resident call on a device copy of the same store:
    I(t) within 1e-3 (the residual projections add their split tiles with
    fp32 atomics, so the last bits vary from run to run), P the exact top-k
    of its own I, and every row that both calls left unselected identical
    in every layer (the stitch).
    Against the oracle (Sink probe, full view): I(t) at 5e-2, the blend
    with this call's P at 2e-2."""
    hs, hreq = _host_store(q3)
    cs = torch.cuda.Stream()
    # the device-resident call runs on a device copy of the same host store
    # (a second chunk prefill would differ in the last bits)
    dK, dV = hs.K.cuda(), hs.V.cuda()
    dsegs = [R.Seg(sg.len, dK[0, hs.where[c.chunk_id][0]], dV[0, hs.where[c.chunk_id][0]],
                   sg.pic_layer_stride, 0) if sg.k_pic is not None else sg
             for sg, c in zip(hreq[0].segs, q3.wl.requests[0].segments)]
    if query is not None and query.get("anchors") == "given":
        # the chunks' anchors kept with the store: no kernel reads the host keys
        anchors, _ = q3.model.cb_anchor_select([sg for sg in dsegs if sg.k_pic is not None],
                                              L.CB_ANCHOR_KNORM, 1000, with_scores=False)
        query = dict(query, anchors=anchors)
    out = q3.model.cb_blend_prefill_host_kv(hreq, 1500, cs, policy=policy, sel_layer=0,
                                            query=query, host_load_ctas=ctas)
    ref = q3.model.cb_blend_prefill([R.Req(hreq[0].tokens, dsegs)], 1500, policy=policy,
                                    sel_layer=0, query=query)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    segs, store = _oracle_inputs(q3)
    N = sum(len(s) for s, c in segs if c)
    k = O.select_count(N, 1500)
    I_h = out["deviation"][:N].cpu().numpy().astype(np.float64)
    I_d = ref["deviation"][:N].cpu().numpy().astype(np.float64)
    assert rms_rel(I_h, I_d) <= 1e-3
    P_h = out["selected"][:k].cpu().numpy()
    assert list(P_h) == list(O.token_topk(I_h, k))
    both = np.setdiff1d(np.arange(N), np.union1d(P_h, ref["selected"][:k].cpu().numpy()))
    rows = torch.from_numpy(both).cuda()
    for l in range(q3.shape.n_layers):
        assert torch.equal(out["k_cache"][l][rows], ref["k_cache"][l][rows]), l
        assert torch.equal(out["v_cache"][l][rows], ref["v_cache"][l][rows]), l
    if rule is None:
        return
    _, I_ref, _ = O.query_probe_select(q3.om, segs, store, 1500, rule, bp, crit)
    assert rms_rel(I_h, I_ref) <= TOL_I
    oref = O.blend_prefill(q3.om, segs, store, 1500, sel_layer=0, forced=P_h)
    for l in range(q3.shape.n_layers):
        assert rms_rel(host(out["k_cache"][l]), oref.K[l]) <= TOL
        assert rms_rel(host(out["v_cache"][l]), oref.V[l]) <= TOL
    Rn = len(oref.rows)
    assert rms_rel(host(out["hidden"][:Rn]), oref.hidden) <= TOL


@pytest.mark.parametrize("policy,query", [
    (L.CB_POLICY_QUERY_PROBE, {"anchor_rule": L.CB_ANCHOR_KNORM, "anchor_bp": 1000,
                               "crit_layers": [1, 2]}),
    (L.CB_POLICY_QUERY_FULL, None),
], ids=["probe_knorm", "full_view"])
def test_query_policies_batch_of_two(q3, policy, query):
    """Two requests in one call (the test request, and its chunks in the
    other order with another query) against each request alone: I(t)
    within 1e-3 (run-to-run rounding of the residual projections), P the
    exact top-k of its own I, and every row left unselected in both calls
    identical in every layer."""
    rng = np.random.default_rng(31)
    rq = q3.wl.requests[0]
    cached = [s for s in rq.segments if s.cached]
    q2 = W.make_tokens(rng, 48, q3.shape.vocab)
    reqs_np = [(list(cached), rq.segments[-1].tokens), (list(reversed(cached)), q2)]
    def gpu_req(chunks, q):
        toks = np.concatenate([s.tokens for s in chunks] + [q]).astype(np.int32)
        return R.Req(torch.from_numpy(toks).cuda(),
                     [q3.store.seg(s.chunk_id) for s in chunks] + [R.Seg(len(q))])
    kw = dict(policy=policy, sel_layer=0, query=query)
    both = q3.model.cb_blend_prefill([gpu_req(*r) for r in reqs_np], 1500, **kw)
    alone = [q3.model.cb_blend_prefill([gpu_req(*r)], 1500, **kw) for r in reqs_np]
    torch.cuda.synchronize()
    assert R.device_status() == 0
    t_off = n_off = k_off = 0
    for (chunks, q), one in zip(reqs_np, alone):
        N = sum(len(s.tokens) for s in chunks)
        T, k = N + len(q), O.select_count(N, 1500)
        I_b = both["deviation"][n_off:n_off + N].cpu().numpy().astype(np.float64)
        I_a = one["deviation"][:N].cpu().numpy().astype(np.float64)
        assert rms_rel(I_b, I_a) <= 1e-3
        P_b = both["selected"][k_off:k_off + k].cpu().numpy()
        assert list(P_b) == list(O.token_topk(I_b, k))
        keep = np.setdiff1d(np.arange(N), np.union1d(P_b, one["selected"][:k].cpu().numpy()))
        rows_b = torch.from_numpy(keep + t_off).cuda()
        rows_a = torch.from_numpy(keep).cuda()
        for l in range(q3.shape.n_layers):
            assert torch.equal(both["k_cache"][l][rows_b], one["k_cache"][l][rows_a]), l
            assert torch.equal(both["v_cache"][l][rows_b], one["v_cache"][l][rows_a]), l
        t_off, n_off, k_off = t_off + T, n_off + N, k_off + k


def test_query_probe_with_given_anchors(q3):
    """A store that keeps each chunk's anchors (cb_anchor_select, Knorm at
    10%) passes them in: the probe then ranks nothing, and its I(t) agrees
    with the call that ranks the same anchors itself (up to the residual
    projections' run-to-run rounding), P the exact top-k of its own I.  An
    anchor outside its chunk is reported as CB_ERR_DEVICE_INDEX."""
    chunks = _chunks(q3)
    segs_g = [q3.store.seg(s.chunk_id) for s in chunks]
    anchors, _ = q3.model.cb_anchor_select(segs_g, L.CB_ANCHOR_KNORM, 1000, with_scores=False)
    base = {"anchor_rule": L.CB_ANCHOR_KNORM, "anchor_bp": 1000, "crit_layers": [1, 2]}
    kw = dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0)
    own = q3.model.cb_blend_prefill(q3.gpu_reqs(), 1500, query=base, **kw)
    given = q3.model.cb_blend_prefill(q3.gpu_reqs(), 1500, query=dict(base, anchors=anchors), **kw)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    N = sum(s.len for s in segs_g)
    k = O.select_count(N, 1500)
    I_o = own["deviation"][:N].cpu().numpy().astype(np.float64)
    I_g = given["deviation"][:N].cpu().numpy().astype(np.float64)
    assert rms_rel(I_g, I_o) <= 1e-3
    assert list(given["selected"][:k].cpu().numpy()) == list(O.token_topk(I_g, k))
    bad = anchors.clone()
    bad[0] = segs_g[0].len                       # one past the first chunk
    q3.model.cb_blend_prefill(q3.gpu_reqs(), 1500, query=dict(base, anchors=bad), **kw)
    torch.cuda.synchronize()
    assert R.device_status() == L.CB_ERR_DEVICE_INDEX


def test_query_probe_knorm_with_the_gpu_anchors(q3):
    chunks = _chunks(q3)
    segs_g = [q3.store.seg(s.chunk_id) for s in chunks]
    anchors, _ = q3.model.cb_anchor_select(segs_g, L.CB_ANCHOR_KNORM, 1000)
    query = {"anchor_rule": L.CB_ANCHOR_KNORM, "anchor_bp": 1000, "crit_layers": [2, 1]}
    out = q3.model.cb_blend_prefill(q3.gpu_reqs(), 1500, policy=L.CB_POLICY_QUERY_PROBE,
                                    sel_layer=0, query=query)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    N = sum(s.len for s in segs_g)
    I_gpu = out["deviation"][:N].cpu().numpy().astype(np.float64)
    # the oracle probes with the GPU's anchors (a float decision on bf16 keys)
    a = anchors.cpu().numpy().astype(np.int64)
    glob, off_a, off_c = [], 0, 0
    for s in segs_g:
        cnt = O.anchor_count(s.len, 1000)
        glob.append(a[off_a:off_a + cnt] + off_c)
        off_a += cnt
        off_c += s.len
    glob = np.concatenate(glob)
    segs, store = _oracle_inputs(q3)
    m = q3.om
    K = np.concatenate([np.stack([O.reposition_keys(kc[l], o, m.n_kv_heads, m.head_dim,
                                                    m.rope_base) for l in range(m.n_layers)])
                        for (kc, _), o in zip(store, np.cumsum([0] + [s.len for s in segs_g])[:-1])],
                       1)
    V = np.concatenate([np.asarray(vc) for _, vc in store], 1)
    u = segs[-1][0]
    I_ref = O.query_probe_scores(m, u, N + np.arange(len(u)), K, V, glob, [1, 2])
    assert rms_rel(I_gpu, I_ref) <= TOL_I


def test_query_policies_validate(q3):
    reqs = q3.gpu_reqs()
    bad = [
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=1,
             query={"anchor_rule": 0, "anchor_bp": 1000, "crit_layers": [1]}),
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0,
             query={"anchor_rule": 0, "anchor_bp": 1000, "crit_layers": [3]}),
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0,
             query={"anchor_rule": 0, "anchor_bp": 1000, "crit_layers": [1, 1]}),
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0,
             query={"anchor_rule": 0, "anchor_bp": 1000, "crit_layers": []}),
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0,
             query={"anchor_rule": 2, "anchor_bp": 1000, "crit_layers": [1]}),
        dict(policy=L.CB_POLICY_QUERY_PROBE, sel_layer=0,
             query={"anchor_rule": 0, "anchor_bp": 10001, "crit_layers": [1]}),
    ]
    for kw in bad:
        with pytest.raises(L.CBError) as e:
            q3.model.plan(reqs, 1500, **kw)
        assert e.value.status == L.CB_ERR_INVALID_ARG
