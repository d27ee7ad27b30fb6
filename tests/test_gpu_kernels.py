"""Kernel-level parity of the CUDA path (through the C ABI) against the CPU
oracle, brute force and exact definitions, on seeded inputs.  Sizes span
several tiles with ragged tails, plus the full sizes of the workloads."""
import ctypes as C
import math

import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L
from gpu_common import (assert_close, bf16_values, dev, host, rms_rel)

pytestmark = pytest.mark.gpu
DTYPES = [torch.float32, torch.bfloat16]


def _vals(rng, shape, dt, std=1.0):
    x = (rng.standard_normal(shape) * std).astype(np.float32)
    return bf16_values(x) if dt == torch.bfloat16 else x


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.synchronize()
    R.device_status()          # read-and-clear before each test
    yield


# ------------------------------------------------------------------ RoPE --
def test_rope_table_matches_definition():
    for hd, base, P in [(64, 1e4, 1000), (128, 1e4, 40000), (128, 5e5, 300)]:
        t = host(R.cb_rope_table_init(P, hd, base)).reshape(P, hd // 2, 2)
        ang = np.multiply.outer(np.arange(P, dtype=np.float64), O.rope_inv_freq(hd, base))
        np.testing.assert_allclose(t[..., 0], np.cos(ang), atol=2e-7)
        np.testing.assert_allclose(t[..., 1], np.sin(ang), atol=2e-7)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("hd,Hkv", [(64, 2), (128, 8)])
def test_reposition_matches_oracle(dt, hd, Hkv):
    rng = np.random.default_rng(1)
    n_layers, kvw = 3, Hkv * hd
    lens = [37, 128, 1, 250]
    deltas = [0, 37, 165, -20]            # rotation per chunk
    dst = [5, 42, 170, 171]
    T = 430
    table = R.cb_rope_table_init(4096, hd, 1e4)
    chunks = [(_vals(rng, (n_layers, n, kvw), dt), _vals(rng, (n_layers, n, kvw), dt))
              for n in lens]
    dk = [(dev(k, dt), dev(v, dt)) for k, v in chunks]
    kc = torch.full((n_layers, T, kvw), 7.0, dtype=dt, device="cuda")
    vc = torch.full_like(kc, 7.0)
    descs = [(k, v, n * kvw, n, d0, de) for (k, v), n, d0, de in zip(dk, lens, dst, deltas)]
    R.cb_rope_reposition(descs, 1, 3, kc, vc, T * kvw, kvw, hd, table, 4096)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    K, V = host(kc), host(vc)
    covered = np.zeros(T, bool)
    for (k, v), n, d0, de in zip(chunks, lens, dst, deltas):
        covered[d0:d0 + n] = True
        for l in (1, 2):
            ref = O.reposition_keys(k[l].astype(np.float64), de, Hkv, hd, 1e4)
            assert_close(K[l, d0:d0 + n], ref, dt)
            assert np.array_equal(V[l, d0:d0 + n], v[l])            # values copied
            if de == 0:
                assert np.array_equal(K[l, d0:d0 + n], k[l])       # identity
    assert np.all(K[0] == 7.0) and np.all(V[0] == 7.0)             # layer 0 untouched
    assert np.all(K[1:, ~covered] == 7.0)                           # other rows untouched


def test_reposition_composes_rotations():
    # rotating by a then by b equals rotating by a+b (RoPE composition)
    rng = np.random.default_rng(2)
    hd, kvw, n = 128, 256, 64
    table = R.cb_rope_table_init(40000, hd, 1e4)
    k0 = dev(_vals(rng, (1, n, kvw), torch.float32))
    v0 = torch.zeros_like(k0)
    a = torch.empty_like(k0); b = torch.empty_like(k0); c = torch.empty_like(k0)
    R.cb_rope_reposition([(k0, v0, n * kvw, n, 0, 3000)], 0, 1, a, torch.empty_like(a), n * kvw, kvw, hd, table, 40000)
    R.cb_rope_reposition([(a, v0, n * kvw, n, 0, 29000)], 0, 1, b, torch.empty_like(b), n * kvw, kvw, hd, table, 40000)
    R.cb_rope_reposition([(k0, v0, n * kvw, n, 0, 32000)], 0, 1, c, torch.empty_like(c), n * kvw, kvw, hd, table, 40000)
    np.testing.assert_allclose(host(b), host(c), atol=2e-4)


# -------------------------------------------------- deviation and top-k --
def _sel_call(kf, kr, reqs, policy=L.CB_POLICY_TOKEN_TOPK):
    n_total = sum(r["n_ctx"] for r in reqs)
    k_total = sum(r["k"] for r in reqs)
    d = torch.empty(max(n_total, 1), dtype=torch.float32, device="cuda")
    idx = torch.full((max(k_total, 1),), -1, dtype=torch.int32, device="cuda")
    R.cb_kv_deviation_topk(kf, kr, reqs, policy, d, idx)
    torch.cuda.synchronize()
    return d.cpu().numpy(), idx.cpu().numpy()


@pytest.mark.parametrize("dt", DTYPES)
def test_deviation_and_topk_small(dt):
    rng = np.random.default_rng(3)
    kvw = 256
    Ns, ks = [300, 1, 1000, 64, 17], [45, 1, 1000, 0, 16]
    rows = sum(Ns) + 50
    kf = _vals(rng, (rows, kvw), dt)
    kr = _vals(rng, (rows + 10, kvw), dt)
    # adversarial ties: identical rows -> d = 0, duplicated differences
    kr[10:40] = kf[10:40]
    kr[500:600] = kf[500:600] + 0.5
    if dt == torch.bfloat16:
        kr = bf16_values(kr)                      # the values the GPU sees
    reqs, f0, doff, ioff = [], 3, 0, 0
    for n, k in zip(Ns, ks):
        reqs.append(dict(n_ctx=n, k=k, fresh_row0=f0, reused_row0=f0 + 7,
                         dev_offset=doff, idx_offset=ioff))
        f0 += n; doff += n; ioff += k
    d, idx = _sel_call(dev(kf, dt), dev(kr, dt), reqs)
    io = 0
    for r in reqs:
        n, k = r["n_ctx"], r["k"]
        a, b = r["fresh_row0"], r["reused_row0"]
        ref = O.kv_deviation(kf[a:a + n].astype(np.float64), kr[b:b + n].astype(np.float64))
        gd = d[r["dev_offset"]:r["dev_offset"] + n]
        np.testing.assert_allclose(gd, ref, rtol=1e-5, atol=1e-6)
        # bit-exact selection against a full sort of the GPU's own d
        assert list(idx[io:io + k]) == list(O.token_topk(gd.astype(np.float64), k))
        io += k


@pytest.mark.parametrize("n,k,B", [(10240, 3072, 4), (32768, 9830, 2), (32768, 1638, 2),
                                   (3072, 460, 1), (7600, 380, 1)])
def test_topk_at_workload_sizes(n, k, B):
    rng = np.random.default_rng(n + k)
    kvw = 1024
    kf = _vals(rng, (n * B, kvw), torch.bfloat16)
    kr = _vals(rng, (n * B, kvw), torch.bfloat16)
    kr[: n // 3] = kf[: n // 3]                       # a block of exact zeros
    reqs = [dict(n_ctx=n, k=k, fresh_row0=b * n, reused_row0=b * n, dev_offset=b * n,
                 idx_offset=b * k) for b in range(B)]
    d, idx = _sel_call(dev(kf, torch.bfloat16), dev(kr, torch.bfloat16), reqs)
    for b in range(B):
        gd = d[b * n:(b + 1) * n].astype(np.float64)
        ref = np.lexsort((np.arange(n), -gd))[:k]
        assert np.array_equal(idx[b * k:(b + 1) * k], np.sort(ref))
    # sampled deviation rows against the definition
    for i in rng.choice(n * B, 64, replace=False):
        ref = np.sum((kf[i].astype(np.float64) - kr[i]) ** 2)
        assert abs(d[i] - ref) <= 1e-5 * ref + 1e-6


def test_doc_aligned_matches_oracle():
    rng = np.random.default_rng(5)
    kvw = 64
    cases = []
    # integer deviations (rows of 0/1 against zero) give exact ties
    for trial in range(40):
        m = int(rng.integers(1, 12))
        lens = rng.integers(0, 60, size=m)
        offs = [0] + list(np.cumsum(lens))
        n = offs[-1]
        if n == 0:
            continue
        k = int(rng.integers(1, n + 1))
        cases.append((offs, n, k, trial % 2 == 0))
    for offs, n, k, integer in cases:
        if integer:
            kf = (rng.random((n, kvw)) < 0.1).astype(np.float32)
        else:
            kf = rng.standard_normal((n, kvw)).astype(np.float32)
        kr = np.zeros_like(kf)
        d, idx = _sel_call(dev(kf), dev(kr), [dict(n_ctx=n, k=k, span_offsets=offs)],
                           L.CB_POLICY_DOC_ALIGNED)
        ref = O.doc_aligned_select(d[:n].astype(np.float64), offs, k)
        assert list(idx[:k]) == list(ref), (offs, k)


def test_doc_aligned_rolling_shape():
    # 19 cached 400-token documents, k = 380 (5%): a window in the top document
    rng = np.random.default_rng(6)
    n, kvw = 7600, 1024
    kf = bf16_values(rng.standard_normal((n, kvw)).astype(np.float32))
    kr = bf16_values(kf + (rng.standard_normal((n, kvw)) * 0.3).astype(np.float32))
    offs = list(range(0, n + 1, 400))
    d, idx = _sel_call(dev(kf, torch.bfloat16), dev(kr, torch.bfloat16),
                       [dict(n_ctx=n, k=380, span_offsets=offs)], L.CB_POLICY_DOC_ALIGNED)
    ref = O.doc_aligned_select(d[:n].astype(np.float64), offs, 380)
    assert list(idx[:380]) == list(ref)
    assert idx[379] - idx[0] == 379                           # one contiguous window


def test_span_policy_controls_match_oracle():
    """"Request Order Matters" §2.3 / §4.4 controls and EPIC's first-token
    rule, each exactly against the oracle on the GPU's own deviations;
    integer-valued deviations in half of the cases give exact ties."""
    rng = np.random.default_rng(15)
    kvw = 64
    for trial in range(30):
        m = int(rng.integers(1, 10))
        lens = rng.integers(0, 50, size=m)
        offs = [0] + [int(x) for x in np.cumsum(lens)]
        n = offs[-1]
        if n == 0:
            continue
        k = int(rng.integers(1, n + 1))
        if trial % 2 == 0:
            kf = (rng.random((n, kvw)) < 0.1).astype(np.float32)
        else:
            kf = rng.standard_normal((n, kvw)).astype(np.float32)
        kr = np.zeros_like(kf)
        order = [int(x) for x in rng.permutation(m)]
        L_, off_ = int(rng.integers(1, 40)), 0
        off_ = int(rng.integers(0, L_ + 1))
        cases = [
            (L.CB_POLICY_SINGLE_WINDOW, dict(), lambda d: O.single_window_select(d, k)),
            (L.CB_POLICY_FIXED_CHUNK, dict(span_len=L_, span_offset=off_),
             lambda d: O.doc_aligned_select(d, O.fixed_chunk_offsets(n, L_, off_), k)),
            (L.CB_POLICY_RANDOM_DOC, dict(span_offsets=offs, span_order=order),
             lambda d: O.doc_aligned_select(d, offs, k, order=order)),
            (L.CB_POLICY_FIRST_TOKENS, dict(span_offsets=offs),
             lambda d: O.first_tokens_select(offs, k)),
        ]
        for policy, extra, ref_fn in cases:
            d, idx = _sel_call(dev(kf), dev(kr), [dict(n_ctx=n, k=k, **extra)], policy)
            ref = ref_fn(d[:n].astype(np.float64))
            assert list(idx[:k]) == list(ref), (policy, offs, k)


def test_span_policies_rolling_shape():
    # 19 cached 400-token documents, k = 380 (5%); fixed 92-token spans
    rng = np.random.default_rng(16)
    n, kvw, k = 7600, 1024, 380
    kf = bf16_values(rng.standard_normal((n, kvw)).astype(np.float32))
    kr = bf16_values(kf + (rng.standard_normal((n, kvw)) * 0.3).astype(np.float32))
    offs = list(range(0, n + 1, 400))
    order = [int(x) for x in rng.permutation(19)]
    for policy, extra, ref_fn in (
            (L.CB_POLICY_SINGLE_WINDOW, dict(), lambda d: O.single_window_select(d, k)),
            (L.CB_POLICY_FIXED_CHUNK, dict(span_len=92, span_offset=46),
             lambda d: O.doc_aligned_select(d, O.fixed_chunk_offsets(n, 92, 46), k)),
            (L.CB_POLICY_RANDOM_DOC, dict(span_offsets=offs, span_order=order),
             lambda d: O.doc_aligned_select(d, offs, k, order=order)),
            (L.CB_POLICY_FIRST_TOKENS, dict(span_offsets=offs),
             lambda d: O.first_tokens_select(offs, k))):
        d, idx = _sel_call(dev(kf, torch.bfloat16), dev(kr, torch.bfloat16),
                           [dict(n_ctx=n, k=k, **extra)], policy)
        assert list(idx[:k]) == list(ref_fn(d[:n].astype(np.float64))), policy
        assert O.selection_segments(idx[:k]) >= 1


def test_span_policy_arguments_are_validated():
    kf = torch.zeros(10, 64, device="cuda")
    bad = [
        (L.CB_POLICY_RANDOM_DOC, dict(n_ctx=10, k=3, span_offsets=[0, 5, 10], span_order=[0, 0])),
        (L.CB_POLICY_RANDOM_DOC, dict(n_ctx=10, k=3, span_offsets=[0, 5, 10])),
        (L.CB_POLICY_FIXED_CHUNK, dict(n_ctx=10, k=3, span_len=0)),
        (L.CB_POLICY_FIXED_CHUNK, dict(n_ctx=10, k=3, span_len=4, span_offset=5)),
        (L.CB_POLICY_FIRST_TOKENS, dict(n_ctx=10, k=3, span_offsets=[0, 5, 9])),
    ]
    for policy, r in bad:
        with pytest.raises(L.CBError):
            R.cb_kv_deviation_topk(kf, kf, [r], policy, torch.empty(10, device="cuda"),
                                   torch.empty(10, dtype=torch.int32, device="cuda"))


# ------------------------------------------------------- gather / scatter --
@pytest.mark.parametrize("dt", DTYPES)
def test_gather_scatter_exact(dt):
    rng = np.random.default_rng(7)
    src = _vals(rng, (500, 1024), dt)
    idx = rng.choice(500, 77, replace=False).astype(np.int32)
    ts = dev(src, dt)
    out = torch.empty(77, 1024, dtype=dt, device="cuda")
    R.cb_gather_rows(ts, dev(idx, torch.int32), out)
    assert np.array_equal(host(out), src[idx])
    kc = torch.zeros(600, 1024, dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    rows = np.sort(rng.choice(600, 77, replace=False)).astype(np.int32)
    R.cb_scatter_kv(out, out * 2, dev(rows, torch.int32), kc, vc)
    K, V = host(kc), host(vc)
    assert np.array_equal(K[rows], src[idx]) and np.array_equal(V[rows], 2 * src[idx].astype(np.float64))
    rest = np.setdiff1d(np.arange(600), rows)
    assert np.all(K[rest] == 0) and np.all(V[rest] == 0)
    torch.cuda.synchronize()
    assert R.device_status() == 0


def test_out_of_range_index_is_reported_not_faulted():
    src = torch.zeros(10, 64, device="cuda")
    out = torch.zeros(3, 64, device="cuda")
    R.cb_gather_rows(src, torch.tensor([1, 10, 2], dtype=torch.int32, device="cuda"), out)
    assert R.device_status() == L.CB_ERR_DEVICE_INDEX
    assert R.device_status() == 0                              # read clears it


def test_bounded_wait_expires_with_status():
    R.cb_debug_expire_wait(2000)
    assert R.device_status() == L.CB_ERR_TIMEOUT
    x = torch.ones(4, device="cuda") * 3                          # context still usable
    assert float(x.sum()) == 12.0


# --------------------------------------------------------------- attention --
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("Hq,Hkv,hd", [(4, 2, 64), (32, 8, 128)])
def test_attention_matches_oracle(dt, Hq, Hkv, hd):
    rng = np.random.default_rng(8)
    # the last request's 18 key blocks are split into chunks (and combined)
    Ts = [300, 129, 1, 1100]
    kv0 = [0, 300, 429, 430]
    Ttot = sum(Ts)
    K = _vals(rng, (Ttot, Hkv * hd), dt)
    V = _vals(rng, (Ttot, Hkv * hd), dt)
    pos, reqs, q0 = [], [], 0
    for T, k0, nq in zip(Ts, kv0, [40, 129, 1, 24]):
        p = np.sort(rng.choice(T, nq, replace=False))
        pos.append(p)
        reqs.append((q0, q0 + nq, k0, T))
        q0 += nq
    pos = np.concatenate(pos).astype(np.int32)
    q = _vals(rng, (q0, Hq * hd), dt)
    out = torch.empty(q0, Hq * hd, dtype=dt, device="cuda")
    R.cb_sparse_query_attention(dev(q, dt), dev(pos, torch.int32), reqs, dev(K, dt), dev(V, dt),
                                Hq, Hkv, hd, out)
    got = host(out)
    for (qb, qe, k0, T) in reqs:
        ref = O.causal_attention(q[qb:qe].reshape(-1, Hq, hd).astype(np.float64), pos[qb:qe],
                                 K[k0:k0 + T].reshape(T, Hkv, hd).astype(np.float64),
                                 V[k0:k0 + T].reshape(T, Hkv, hd).astype(np.float64), Hq, Hkv)
        assert_close(got[qb:qe], ref.reshape(qe - qb, -1), dt)
    assert R.device_status() == 0


# ------------------------------------------------------------------ GEMM --
def _small_model(dt_name, d=256, F=688, Hq=4, Hkv=2, hd=64):
    shape = W.ModelShape("t", 1, d, Hq, Hkv, hd, F, 512, dtype=dt_name)
    w = W.make_weights(shape, 11)
    return shape, w, R.BlendModel.from_host(shape, w, 1024)


@pytest.mark.parametrize("dt_name", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 77, 300])
def test_linear_epilogues(dt_name, M):
    shape, w, model = _small_model(dt_name)
    dt = model.dtype
    rng = np.random.default_rng(M)
    A = _vals(rng, (M, shape.d_model), dt)
    lw = w["layers"][0]
    Wq = lw["w_qkv"].astype(np.float64)
    out = torch.empty(M, Wq.shape[0], dtype=dt, device="cuda")
    model.cb_linear(dev(A, dt), model.w["layers"][0]["w_qkv"], out, L.CB_EPI_STORE)
    assert_close(host(out), A.astype(np.float64) @ Wq.T, dt)
    h0 = rng.standard_normal((M, shape.d_model)).astype(np.float32)
    h = dev(h0)
    Ao = _vals(rng, (M, shape.n_q_heads * shape.head_dim), dt)
    model.cb_linear(dev(Ao, dt), model.w["layers"][0]["w_o"], h, L.CB_EPI_RESID)
    ref = h0 + Ao.astype(np.float64) @ lw["w_o"].astype(np.float64).T
    assert_close(host(h), ref, torch.float32 if dt == torch.float32 else dt)
    g = torch.empty(M, shape.d_ffn, dtype=dt, device="cuda")
    model.cb_linear(dev(A, dt), model.w["layers"][0]["w_gate"], g, L.CB_EPI_SWIGLU,
                    W2=model.w["layers"][0]["w_up"])
    A64 = A.astype(np.float64)
    ref = O.silu(A64 @ lw["w_gate"].astype(np.float64).T) * (A64 @ lw["w_up"].astype(np.float64).T)
    assert_close(host(g), ref, dt)


@pytest.fixture
def gemm_path(request):
    R.cb_debug_gemm_path(request.param)
    yield request.param
    R.cb_debug_gemm_path(L.CB_GEMM_AUTO)


@pytest.mark.parametrize("gemm_path", [L.CB_GEMM_TOKEN_M, L.CB_GEMM_SWAP_AB,
                                       L.CB_GEMM_SWAP_AB_PAIR], indirect=True)
@pytest.mark.parametrize("M", [524, 128, 3136, 1])
def test_tensor_core_gemm_llama_shapes(M, gemm_path):
    """bf16 tcgen05 GEMMs (token rows on M, and the swapped form) at the
    workload's projection shapes: ragged M, stream-K residual over
    K = 14336, SwiGLU over N = 14336."""
    rng = np.random.default_rng(M)
    shape = W.ModelShape("g", 1, 4096, 32, 8, 128, 14336, 256, dtype="bf16")
    w = {"embed": np.zeros((256, 4096), np.float32),
         "final_norm": np.ones(4096, np.float32),
         "layers": [{
             "w_qkv": _vals(rng, (6144, 4096), torch.bfloat16, 0.02),
             "w_o": _vals(rng, (4096, 4096), torch.bfloat16, 0.02),
             "w_gate": _vals(rng, (14336, 4096), torch.bfloat16, 0.02),
             "w_up": _vals(rng, (14336, 4096), torch.bfloat16, 0.02),
             "w_down": _vals(rng, (4096, 14336), torch.bfloat16, 0.02),
             "norm1": np.ones(4096, np.float32), "norm2": np.ones(4096, np.float32)}]}
    model = R.BlendModel.from_host(shape, w, 1024)
    lw = w["layers"][0]
    dw = model.w["layers"][0]
    A = _vals(rng, (M, 4096), torch.bfloat16)
    A64 = A.astype(np.float64)
    out = torch.empty(M, 6144, dtype=torch.bfloat16, device="cuda")
    model.cb_linear(dev(A, torch.bfloat16), dw["w_qkv"], out, L.CB_EPI_STORE)
    ref = A64 @ lw["w_qkv"].astype(np.float64).T
    assert rms_rel(host(out), ref) < 5e-3
    G = _vals(rng, (M, 14336), torch.bfloat16)
    h0 = rng.standard_normal((M, 4096)).astype(np.float32)
    h = dev(h0)
    model.cb_linear(dev(G, torch.bfloat16), dw["w_down"], h, L.CB_EPI_RESID)
    ref = h0 + G.astype(np.float64) @ lw["w_down"].astype(np.float64).T
    assert rms_rel(host(h), ref) < 5e-5      # fp32 accumulation over K = 14336
    g = torch.empty(M, 14336, dtype=torch.bfloat16, device="cuda")
    model.cb_linear(dev(A, torch.bfloat16), dw["w_gate"], g, L.CB_EPI_SWIGLU, W2=dw["w_up"])
    ref = O.silu(A64 @ lw["w_gate"].astype(np.float64).T) * (A64 @ lw["w_up"].astype(np.float64).T)
    assert rms_rel(host(g), ref) < 5e-3
    torch.cuda.synchronize()
    assert R.device_status() == 0


@pytest.fixture(scope="module")
def llama_proj():
    rng = np.random.default_rng(7)
    shape = W.ModelShape("g", 1, 4096, 32, 8, 128, 14336, 256, dtype="bf16")
    w = {"embed": np.zeros((256, 4096), np.float32),
         "final_norm": np.ones(4096, np.float32),
         "layers": [{
             "w_qkv": _vals(rng, (6144, 4096), torch.bfloat16, 0.02),
             "w_o": _vals(rng, (4096, 4096), torch.bfloat16, 0.02),
             "w_gate": _vals(rng, (14336, 4096), torch.bfloat16, 0.02),
             "w_up": _vals(rng, (14336, 4096), torch.bfloat16, 0.02),
             "w_down": _vals(rng, (4096, 14336), torch.bfloat16, 0.02),
             "norm1": np.ones(4096, np.float32), "norm2": np.ones(4096, np.float32)}]}
    return w, R.BlendModel.from_host(shape, w, 1024)


@pytest.mark.parametrize("gemm_path", [L.CB_GEMM_SWAP_AB, L.CB_GEMM_SWAP_AB_PAIR], indirect=True)
@pytest.mark.parametrize("M", [524, 128, 3136, 1])
def test_gemm_tail_split(M, gemm_path, llama_proj):
    """The swapped GEMM with the tail-split workspace.  At these shapes the
    tiles of the partial last wave run as 2 to 9 k-segments on otherwise idle
    SMs (SwiGLU over N = 14336 at every M; the N = 6144 projection at 128,
    3136 and 1 rows); segment 0 adds the others' fp32 partials in segment
    order.  Checked: the oracle's product, bit-identical repeats, and the
    unsplit launch up to fp32 summation order."""
    w, model = llama_proj
    lw = w["layers"][0]
    dw = model.w["layers"][0]
    rng = np.random.default_rng(100 + M)
    A = _vals(rng, (M, 4096), torch.bfloat16)
    A64 = A.astype(np.float64)
    Ad = dev(A, torch.bfloat16)
    ws = torch.empty(L.lib.cb_linear_workspace_size(), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)            # the call needs no initialised workspace
    outs = []
    for _ in range(2):
        out = torch.empty(M, 6144, dtype=torch.bfloat16, device="cuda")
        model.cb_linear_ws(Ad, dw["w_qkv"], out, L.CB_EPI_STORE, ws=ws)
        g = torch.empty(M, 14336, dtype=torch.bfloat16, device="cuda")
        model.cb_linear_ws(Ad, dw["w_gate"], g, L.CB_EPI_SWIGLU, W2=dw["w_up"], ws=ws)
        outs.append((out, g))
    torch.cuda.synchronize()
    assert R.device_status() == 0
    ref = A64 @ lw["w_qkv"].astype(np.float64).T
    assert rms_rel(host(outs[0][0]), ref) < 5e-3
    ref = O.silu(A64 @ lw["w_gate"].astype(np.float64).T) * (A64 @ lw["w_up"].astype(np.float64).T)
    assert rms_rel(host(outs[0][1]), ref) < 5e-3
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # the unsplit launch: the same sums in another fp32 order
    g1 = torch.empty(M, 14336, dtype=torch.bfloat16, device="cuda")
    model.cb_linear(Ad, dw["w_gate"], g1, L.CB_EPI_SWIGLU, W2=dw["w_up"])
    torch.cuda.synchronize()
    assert rms_rel(host(outs[0][1]), host(g1)) < 2e-3


@pytest.fixture
def mlp_fusion():
    yield
    L.check(L.lib.cb_debug_mlp_fusion(1))


@pytest.mark.parametrize("gemm_path", [L.CB_GEMM_AUTO, L.CB_GEMM_SWAP_AB], indirect=True)
@pytest.mark.parametrize("M", [524, 64, 300, 3136, 9])
def test_fused_mlp_layer_matches_two_launches(M, gemm_path, llama_proj, mlp_fusion):
    """One bf16 decoder layer (cb_blend_layer, M rows attending causally over
    themselves) with the MLP as one launch (gate/up + SwiGLU, then the down
    projection waiting per k-block on the gate/up tiles' flags) and as two.
    The K/V the layer scatters precede the MLP and match bit for bit; the
    layer's update of h matches up to fp32 summation order (split gate/up
    tiles; the residual adds' order, which can move a bf16 rounding of the
    normalised rows: about 2e-4 between repeats at 64 rows); the launch probe
    sees one fused launch.  The workspace is filled with 0xFF bytes before
    every call (NaN in the gate/up output, -1 in every flag), so a down
    k-block read before its gate/up tile wrote it, or a flag not reset by
    the call, shows as a non-finite h.  9 rows: the single-CTA form."""
    w, model = llama_proj
    rng = np.random.default_rng(300 + M)
    h0 = dev(rng.standard_normal((M, 4096)).astype(np.float32))
    pos = torch.arange(M, dtype=torch.int32, device="cuda")
    reqs = [(0, M, 0, M)]
    ws = torch.empty(max(L.lib.cb_layer_workspace_size(model.handle, M), 256), dtype=torch.uint8,
                     device="cuda")
    res = {}
    for fused in (1, 0, 1):
        L.check(L.lib.cb_debug_mlp_fusion(fused))
        h = h0.clone()
        kc = torch.zeros(M, 1024, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        ws.fill_(0xFF)
        L.check(L.lib.cb_debug_probe_start(L.CB_PROBE_MLP, 4))
        model.cb_blend_layer(0, h, pos, pos, reqs, kc, vc, ws=ws)
        n = C.c_int()
        ms = C.c_float()
        L.check(L.lib.cb_debug_probe_stop(C.byref(n), C.byref(ms)))
        assert n.value == fused
        res.setdefault(fused, []).append((h, kc, vc))
    torch.cuda.synchronize()
    assert R.device_status() == 0
    (hf, kf, vf), (hf2, _, _) = res[1]
    hu, ku, vu = res[0][0]
    assert torch.equal(kf, ku) and torch.equal(vf, vu)
    d_f, d_u, d_f2 = host(hf) - host(h0), host(hu) - host(h0), host(hf2) - host(h0)
    assert np.isfinite(d_f).all() and np.isfinite(d_f2).all() and np.isfinite(d_u).all()
    assert rms_rel(d_f, d_u) < 2e-3
    assert rms_rel(d_f2, d_f) < 2e-3


def test_linear_workspace_is_validated(llama_proj):
    w, model = llama_proj
    dw = model.w["layers"][0]
    A = torch.zeros(8, 4096, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(8, 6144, dtype=torch.bfloat16, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(L.CBError) as e:
        model.cb_linear_ws(A, dw["w_qkv"], out, L.CB_EPI_STORE, ws=small)
    assert e.value.status == L.CB_ERR_WORKSPACE


def test_selection_stats_match_the_definitions():
    """cb_selection_stats against the oracle's Table 2 definitions ("Request
    Order Matters" §4.4): contiguous regions of a selection and the share of
    the deviation it carries, on random requests, several per call."""
    import ctypes as C
    rng = np.random.default_rng(0)
    for trial in range(10):
        reqs, ds, Ps, d_off, i_off = [], [], [], 0, 0
        for b in range(int(rng.integers(1, 5))):
            n = int(rng.integers(1, 3000))
            d = rng.random(n).astype(np.float32)
            k = int(rng.integers(0, n + 1))
            P = np.sort(rng.choice(n, size=k, replace=False)).astype(np.int32)
            reqs.append(dict(n_ctx=n, k=k, dev_offset=d_off, idx_offset=i_off))
            ds.append(d); Ps.append(P)
            d_off += n; i_off += k
        dev = torch.from_numpy(np.concatenate(ds)).cuda()
        idx = torch.from_numpy(np.concatenate(Ps + [np.zeros(1, np.int32)])).cuda()
        seg = torch.full((len(reqs),), -1, dtype=torch.int32, device="cuda")
        cap = torch.full((len(reqs),), -1.0, dtype=torch.float64, device="cuda")
        arr, keep = R.api._select_reqs(reqs)
        L.check(L.lib.cb_selection_stats(C.c_void_p(dev.data_ptr()), C.c_void_p(idx.data_ptr()),
                                         arr, len(reqs), C.c_void_p(seg.data_ptr()),
                                         C.c_void_p(cap.data_ptr()),
                                         C.c_void_p(torch.cuda.current_stream().cuda_stream)))
        torch.cuda.synchronize()
        assert R.device_status() == 0
        for b, (d, P) in enumerate(zip(ds, Ps)):
            assert int(seg[b]) == O.selection_segments(P)
            assert abs(float(cap[b]) - O.captured_deviation(P, d.astype(np.float64))) < 1e-9
    # the single-request binding
    s_, c_ = R.selection_stats(torch.tensor([3, 4, 5, 9], dtype=torch.int32, device="cuda"),
                               torch.ones(12, dtype=torch.float32, device="cuda"))
    assert (s_, c_) == (2, 4 / 12)
