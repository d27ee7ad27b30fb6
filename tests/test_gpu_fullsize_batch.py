"""Full-size sampled parity for the batched workloads (see fullsize_common):

* the Qwen3-8B-shaped stack (36 layers, F = 12288), 4 independent requests,
  each 10 chunks drawn in a seeded order from a shared pool of 40 x 1024
  tokens + 128 query tokens, 30% token top-k;
* the 32K long-context batch on the Llama-3-8B shape (2 x 32 chunks x 1024
  + 256 query tokens) at r = 5, 10, 20 and 30%.

Per request: sampled rows against the oracle, the selection exactly the
top-k of the GPU's own deviations, unselected rows of every layer >= 1 bit
for bit the pure stitch (a r = 0 call), and the first token the arg-max of
the tied head on the final hidden state."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import rag_kv_cache_layer_gb300 as R
from fullsize_common import check_request, oracle_model, sampled_reference
from gpu_common import rms_rel

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _setup(wl, seed, max_pos):
    dev = torch.device("cuda", 0)
    shape = wl.model
    model = R.BlendModel(shape, W.make_weights_device(shape, seed, dev), max_pos, dev)
    cached = {}
    for rq in wl.requests:
        for sg in rq.segments:
            if sg.cached:
                cached[sg.chunk_id] = sg.tokens
    store = R.ChunkStore(model, sum(len(t) for t in cached.values()))
    store.prefill({c: torch.from_numpy(t).to(dev) for c, t in cached.items()})
    reqs = [R.Req(torch.from_numpy(rq.tokens).to(dev),
                  [store.seg(sg.chunk_id) if sg.cached else R.Seg(len(sg.tokens))
                   for sg in rq.segments]) for rq in wl.requests]
    torch.cuda.synchronize()
    return model, store, reqs


def _offsets(wl, ratio_bp):
    T = [rq.n_tokens for rq in wl.requests]
    N = [rq.n_ctx for rq in wl.requests]
    k = [O.select_count(n, ratio_bp) for n in N]
    cs = lambda a: np.concatenate([[0], np.cumsum(a)]).astype(int)
    return T, N, k, cs(T), cs(N), cs(k)


def _samples(rq, sel, rng):
    lens = [len(sg.tokens) for sg in rq.segments if sg.cached]
    offs = np.cumsum([0] + lens)
    picks = {0, 5, int(offs[1]) - 1, int(offs[1]), int(offs[-2]), rq.n_ctx - 1}
    picks |= set(int(x) for x in rng.choice(rq.n_ctx, 3, replace=False))
    picks |= set(int(x) for x in sel[:2]) | set(int(x) for x in sel[-2:])
    return sorted(picks)


def _check_batch(wl, model, reqs, outs, ratio_bp, with_oracle=True):
    T, N, k, t_off, n_off, k_off = _offsets(wl, ratio_bp)
    rng = np.random.default_rng(7)
    shape = wl.model
    L = shape.n_layers
    for b, rq in enumerate(wl.requests):
        d = outs["deviation"][n_off[b]:n_off[b + 1]]
        sel = outs["selected"][k_off[b]:k_off[b + 1]]
        d64 = d.cpu().numpy().astype(np.float64)
        assert list(sel.cpu().numpy()) == list(O.token_topk(d64, k[b]))
        if not with_oracle:
            continue
        m, ids = oracle_model(shape, model.w, rq.tokens)
        samples = _samples(rq, sel.cpu().numpy(), rng)
        ref = sampled_reference(m, ids, [len(sg.tokens) for sg in rq.segments if sg.cached],
                                samples)
        kc = outs["k_cache"][:, t_off[b]:t_off[b + 1]]
        vc = outs["v_cache"][:, t_off[b]:t_off[b + 1]]
        check_request(ref, kc, vc, d, sel, extra_rows=[N[b], T[b] - 1])


def _check_stitch_and_token(wl, model, reqs, outs, ratio_bp):
    T, N, k, t_off, n_off, k_off = _offsets(wl, ratio_bp)
    stitched = model.cb_blend_prefill(reqs, 0)
    torch.cuda.synchronize()
    s = wl.model
    for b in range(len(reqs)):
        keep = torch.ones(N[b], dtype=torch.bool, device="cuda")
        keep[outs["selected"][k_off[b]:k_off[b + 1]].long()] = False
        r0 = t_off[b]
        for l in range(1, s.n_layers):
            a = outs["k_cache"][l][r0:r0 + N[b]][keep]
            assert torch.equal(a, stitched["k_cache"][l][r0:r0 + N[b]][keep])
            a = outs["v_cache"][l][r0:r0 + N[b]][keep]
            assert torch.equal(a, stitched["v_cache"][l][r0:r0 + N[b]][keep])
    del stitched
    # first token of each request: arg-max of the tied head on its last row
    R_off = np.concatenate([[0], np.cumsum([k[b] + T[b] - N[b] for b in range(len(reqs))])])
    E = model.w["embed"]
    for b in range(len(reqs)):
        h = outs["hidden"][int(R_off[b + 1]) - 1].double()
        x = (h / torch.sqrt((h * h).mean() + s.norm_eps)).float()
        logits = torch.cat([E[i:i + 16384].float() @ x for i in range(0, s.vocab, 16384)])
        tok = int(outs["first_token"][b])
        top = float(logits.max())
        assert float(logits[tok]) >= top - 1e-3 * abs(top)


def test_qwen_shaped_batch_of_four():
    wl = W.qwen_pool()
    model, store, reqs = _setup(wl, 2345, 16384)
    outs = model.cb_blend_prefill(reqs, wl.ratio_bp)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    _check_batch(wl, model, reqs, outs, wl.ratio_bp)
    _check_stitch_and_token(wl, model, reqs, outs, wl.ratio_bp)
    assert R.device_status() == 0


def test_long_context_batch_ratio_sweep():
    wl = W.long_context()
    model, store, reqs = _setup(wl, 3456, 40000)
    outs = None
    for i, r in enumerate((500, 1000, 2000, 3000)):
        outs = model.cb_blend_prefill(reqs, r)
        torch.cuda.synchronize()
        assert R.device_status() == 0
        # sampled oracle rows at the smallest budget; exact selection at all
        _check_batch(wl, model, reqs, outs, r, with_oracle=(i == 0))
        if i == 0:
            _check_stitch_and_token(wl, model, reqs, outs, r)
        del outs
    assert R.device_status() == 0
