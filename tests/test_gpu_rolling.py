"""The rolling-agent loop ("Request Order Matters" §4.1) on the CUDA path:
a window of documents whose chunk caches persist in one store while the
oldest is evicted and the newest is prefilled after its request.  Every
request is checked against the oracle (fp32, the 2-layer model): the newest
document is an uncached segment, the others are re-positioned chunk caches,
under both token top-k and document-aligned selection."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L
from gpu_common import assert_close, host, ties_ok

pytestmark = pytest.mark.gpu

WINDOW, DOC, QUERY, N_REQ, RATIO = 5, 24, 8, 5, 2000


@pytest.fixture(scope="module")
def setup():
    shape = W.TINY_F32
    weights = W.make_weights(shape, 0)
    model = R.BlendModel.from_host(shape, weights, 1024)
    om = O.model_from_weights(shape, weights)
    rng = np.random.default_rng(44)
    docs = [W.make_tokens(rng, DOC, shape.vocab) for _ in range(WINDOW + N_REQ - 1)]
    queries = [W.make_tokens(rng, QUERY, shape.vocab) for _ in range(N_REQ)]
    pic = {i: O.chunk_prefill(om, d) for i, d in enumerate(docs)}
    return model, om, docs, queries, pic


@pytest.mark.parametrize("write_back", [False, True])
@pytest.mark.parametrize("policy", [L.CB_POLICY_TOKEN_TOPK, L.CB_POLICY_DOC_ALIGNED])
def test_rolling_window_matches_oracle(setup, policy, write_back):
    """With write_back the store is history dependent ("Request Order
    Matters" §4.2): after every request the cached documents' fused K/V,
    moved back to position 0, replace their stored caches -- on both
    sides, so every later request checks the accumulated state."""
    model, om, docs, queries, pic0 = setup
    pic = dict(pic0)
    dev = lambda a: torch.from_numpy(np.asarray(a, np.int32)).cuda()
    rw = R.RollingWindow(model, WINDOW, DOC, RATIO, policy, write_back=write_back)
    rw.seed({i: dev(docs[i]) for i in range(WINDOW - 1)})
    name = "token_topk" if policy == L.CB_POLICY_TOKEN_TOPK else "doc_aligned"
    for t in range(N_REQ):
        new_id = t + WINDOW - 1
        req = rw.request(dev(docs[new_id]), dev(queries[t]))
        out = rw.blend(req)
        torch.cuda.synchronize()
        assert R.device_status() == 0
        cached = list(range(t, t + WINDOW - 1))
        assert rw.docs == cached
        segs = [(docs[i], True) for i in cached] + [(docs[new_id], False), (queries[t], False)]
        ref = O.blend_prefill(om, segs, [pic[i] for i in cached], RATIO, policy=name)
        k = len(ref.selected)
        sel = out["selected"][:k].cpu().numpy()
        if policy == L.CB_POLICY_TOKEN_TOPK:
            assert ties_ok(sel, ref.selected, ref.deviation, k)
        if set(sel) != set(ref.selected):
            assert not write_back, "the stores would diverge"
        else:                               # else a deviation tie moved the set
            assert_close(host(out["k_cache"]), ref.K, torch.float32)
            assert_close(host(out["v_cache"]), ref.V, torch.float32)
            Rn = len(ref.rows)
            assert np.array_equal(out["rows"][:Rn].cpu().numpy(), ref.rows)
            assert_close(host(out["hidden"][:Rn]), ref.hidden, torch.float32)
        if write_back:
            for cid, kv in zip(cached, O.write_back(ref, segs, om)):
                pic[cid] = kv
            torch.cuda.synchronize()
            for cid in cached:             # the GPU store holds the same state
                r0, n = rw.store.where[cid]
                assert_close(host(rw.store.K[:, r0:r0 + n]), pic[cid][0], torch.float32)
                assert_close(host(rw.store.V[:, r0:r0 + n]), pic[cid][1], torch.float32)
        rw.advance(new_id, dev(docs[new_id]))
    # the store cycles through fixed slots: one window of documents
    assert rw.store.used == (WINDOW - 1) * DOC
