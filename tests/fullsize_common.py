"""Sampled parity at full size: the oracle computes chosen rows of a request
one by one from the (seeded) weights and tokens, with no input taken from
the CUDA path.

For a request of cached chunks followed by uncached tokens:

* layer-0 K/V of every row at its request position (layer 0 sees only the
  row's own embedding, so these are exact for any context);
* for each sampled context row i: the layer-0 output over the request
  prefix, the fresh layer-1 key and value, the chunk-alone (PIC) layer-1 key
  and value moved to the chunk's request offset (QCFuse Eqs. 3-4), and the
  deviation d_i ("Request Order Matters" §2.2 Eq. 1).

The GPU's fused layer-1 row i must then be the fresh K/V if it selected i,
the moved PIC otherwise (QCFuse Eq. 7).
"""
import numpy as np
import torch

import oracle as O
from gpu_common import rms_rel

TOL = 2e-2          # bf16 path against the float64 oracle, RMS-relative


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_model(shape, dev_weights, tokens):
    """A 2-layer float64 oracle model over the request's distinct tokens
    (the embedding holds only those rows; token ids are remapped)."""
    uniq, inv = np.unique(np.asarray(tokens), return_inverse=True)
    idx = torch.from_numpy(uniq.astype(np.int64)).to(dev_weights["embed"].device)
    embed = dev_weights["embed"].index_select(0, idx).float().cpu().numpy()

    def layer(l, keys):
        return {k: f64(dev_weights["layers"][l][k]) for k in keys}
    lw0 = layer(0, ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "norm1", "norm2"))
    lw1 = layer(1, ("w_qkv", "norm1"))
    m = O.Model(2, shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                shape.d_ffn, len(uniq), shape.rope_base, shape.norm_eps, embed,
                np.ones(shape.d_model), [lw0, lw1])
    return m, inv


def sampled_reference(m, tok_ids, chunk_lens, samples):
    """tok_ids: the request's remapped token ids; chunk_lens: lengths of its
    cached chunks, in order; samples: ascending context positions."""
    T = len(tok_ids)
    S = np.asarray(samples, dtype=np.int64)
    pos = np.arange(T)
    E = O.embed_rows(m, tok_ids)
    K0, V0 = O.kv_rows(m, 0, E, pos)              # every row's layer-0 K / V
    h1 = O.decoder_layer(m, 0, E[S], S, K0.copy(), V0.copy(), S, write_kv=False)[0]
    k1f, v1f = O.kv_rows(m, 1, h1, S)
    offs = np.concatenate([[0], np.cumsum(chunk_lens)])
    chunk_of = np.searchsorted(offs, S, side="right") - 1
    local = {}
    for c in np.unique(chunk_of):
        o, jmax = int(offs[c]), int(S[chunk_of == c].max() - offs[c])
        local[c] = O.kv_rows(m, 0, E[o:o + jmax + 1], np.arange(jmax + 1))
    k1p, v1p = np.empty_like(k1f), np.empty_like(v1f)
    for n, i in enumerate(S):
        c = int(chunk_of[n])
        o, j = int(offs[c]), int(i - offs[c])
        K0c, V0c = (a[:j + 1].copy() for a in local[c])
        hc = O.decoder_layer(m, 0, E[[i]], [j], K0c, V0c, [j], write_kv=False)[0]
        kc, vc = O.kv_rows(m, 1, hc, [j])
        k1p[n] = O.reposition_keys(kc, o, m.n_kv_heads, m.head_dim, m.rope_base)[0]
        v1p[n] = vc[0]
    return dict(S=S, K0=K0, V0=V0, k1f=k1f, v1f=v1f, k1p=k1p, v1p=v1p,
                d=O.kv_deviation(k1f, k1p))


def check_request(ref, k_cache, v_cache, deviation, selected, extra_rows=()):
    """k_cache / v_cache: the request's fused cache [layers][T][kvw] (device);
    deviation: its d [N]; selected: its P (device, ascending)."""
    S = ref["S"]
    rows = np.concatenate([S, np.asarray(extra_rows, dtype=np.int64)])
    ix = torch.from_numpy(rows).to(k_cache.device)
    assert rms_rel(f64(k_cache[0][ix]), ref["K0"][rows]) <= TOL
    assert rms_rel(f64(v_cache[0][ix]), ref["V0"][rows]) <= TOL
    d_gpu = deviation[torch.from_numpy(S).to(deviation.device)].cpu().numpy().astype(np.float64)
    assert rms_rel(d_gpu, ref["d"]) <= TOL
    chosen = np.isin(S, selected.cpu().numpy())
    k_ref = np.where(chosen[:, None], ref["k1f"], ref["k1p"])
    v_ref = np.where(chosen[:, None], ref["v1f"], ref["v1p"])
    ix = torch.from_numpy(S).to(k_cache.device)
    assert rms_rel(f64(k_cache[1][ix]), k_ref) <= TOL
    assert rms_rel(f64(v_cache[1][ix]), v_ref) <= TOL
    return d_gpu, chosen


class DeviceLayers:
    """The oracle's per-layer weights, read as float64 from the device tensors
    the GPU runs on (the seeded generator's values), one layer at a time: the
    oracle walks the layers in order, so holding the last layer read keeps
    host memory to one layer (1.75 GB in float64 for the Llama shape)."""

    KEYS = ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "norm1", "norm2")

    def __init__(self, dev_layers):
        self.dev = dev_layers
        self.at, self.cur = None, None
        self.reads = 0

    def __len__(self):
        return len(self.dev)

    def __getitem__(self, l):
        if l != self.at:
            self.cur = {k: self.dev[l][k].double().cpu().numpy() for k in self.KEYS}
            self.at = l
            self.reads += 1
        return self.cur


class DeviceEmbedding:
    """The embedding table as float64 rows fetched on demand (a token list or
    a block of rows); the oracle widens rows where it uses them."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        if isinstance(idx, slice):
            return self.t[idx].double().cpu().numpy()
        ix = np.asarray(idx)
        rows = torch.from_numpy(ix.reshape(-1).astype(np.int64)).to(self.t.device)
        return self.t.index_select(0, rows).double().cpu().numpy().reshape(*ix.shape, -1)


def oracle_model_full(shape, dev_weights):
    """The whole float64 oracle model over the device weights, layers and
    embedding read on demand."""
    return O.Model(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads,
                   shape.head_dim, shape.d_ffn, shape.vocab, shape.rope_base, shape.norm_eps,
                   DeviceEmbedding(dev_weights["embed"]),
                   dev_weights["final_norm"].double().cpu().numpy(),
                   DeviceLayers(dev_weights["layers"]))


def plain_bf16_prefill(shape, dev_weights, tokens):
    """A plain PyTorch bf16 prefill of one standalone token run (positions
    0..n-1): F.linear on bf16 operands, scaled_dot_product_attention in bf16,
    the residual stream in fp32.  It is not the oracle: it measures the
    accumulated rounding of an ordinary bf16 datapath on this model, the
    floor any bf16 implementation is held against at depth.  Returns the
    per-layer K and V rows as float64 numpy [n_layers][n][Hkv*hd]."""
    import torch.nn.functional as F
    dev = dev_weights["embed"].device
    toks = torch.from_numpy(np.asarray(tokens, np.int64)).to(dev)
    n, hd = len(tokens), shape.head_dim
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    inv = shape.rope_base ** (-torch.arange(hd // 2, dtype=torch.float64, device=dev) * 2 / hd)
    ang = torch.arange(n, dtype=torch.float64, device=dev)[:, None] * inv[None]
    cos, sin = torch.cos(ang).float()[:, None], torch.sin(ang).float()[:, None]

    def rope(x):
        a, b = x[..., :hd // 2], x[..., hd // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], -1)

    def norm(h, g):
        return (h / torch.sqrt((h * h).mean(-1, keepdim=True) + shape.norm_eps) * g).to(torch.bfloat16)

    Ks, Vs = [], []
    with torch.no_grad():
        h = dev_weights["embed"][toks].float()
        for L in dev_weights["layers"]:
            qkv = F.linear(norm(h, L["norm1"]), L["w_qkv"]).float()
            q = rope(qkv[:, :Hq * hd].reshape(n, Hq, hd)).to(torch.bfloat16)
            k = rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(n, Hkv, hd)).to(torch.bfloat16)
            v = qkv[:, (Hq + Hkv) * hd:].reshape(n, Hkv, hd).to(torch.bfloat16)
            Ks.append(k.reshape(n, -1).double().cpu().numpy())
            Vs.append(v.reshape(n, -1).double().cpu().numpy())
            o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                               v.transpose(0, 1)[None], is_causal=True,
                                               enable_gqa=True)[0].transpose(0, 1)
            h = h + F.linear(o.reshape(n, -1), L["w_o"]).float()
            x = norm(h, L["norm2"])
            g = F.silu(F.linear(x, L["w_gate"]).float()) * F.linear(x, L["w_up"]).float()
            h = h + F.linear(g.to(torch.bfloat16), L["w_down"]).float()
    return np.stack(Ks), np.stack(Vs)
