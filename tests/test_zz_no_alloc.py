"""cb_kv_deviation_topk_noalloc -- deviation ranking for callers that cannot
allocate device memory (their deviations live in the library's fixed device
array).  Its selections must equal those of cb_kv_deviation_topk, which
takes caller scratch, on two calls in a row with different inputs (a stale
array would show up on the second).  Kept in a file that runs last."""
import numpy as np
import pytest
import torch

import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L

pytestmark = pytest.mark.gpu


def _inputs(seed, kvw=1024):
    rng = np.random.default_rng(seed)
    Ns, ks = [3072, 1000, 17], [460, 1000, 3]
    rows = sum(Ns)
    kf = W.round_to_bf16(rng.standard_normal((rows, kvw)).astype(np.float32))
    kr = W.round_to_bf16(rng.standard_normal((rows, kvw)).astype(np.float32))
    kr[100:140] = kf[100:140]                     # ties at zero deviation
    reqs, r0, io = [], 0, 0
    for n, k in zip(Ns, ks):
        reqs.append(dict(n_ctx=n, k=k, fresh_row0=r0, reused_row0=r0, dev_offset=r0,
                         idx_offset=io, span_offsets=list(range(0, n, 400)) + [n]))
        r0 += n
        io += k
    dev = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16)
    return dev(kf), dev(kr), reqs, sum(ks), rows


@pytest.mark.parametrize("policy", [L.CB_POLICY_TOKEN_TOPK, L.CB_POLICY_DOC_ALIGNED])
def test_noalloc_matches_scratch_version_on_two_calls(policy):
    for seed in (1, 2):                            # two calls in a row
        kf, kr, reqs, k_total, n_total = _inputs(seed)
        ref = torch.full((k_total,), -1, dtype=torch.int32, device="cuda")
        d = torch.empty(n_total, dtype=torch.float32, device="cuda")
        R.cb_kv_deviation_topk(kf, kr, reqs, policy, d, ref)
        got = torch.full((k_total,), -2, dtype=torch.int32, device="cuda")
        R.cb_kv_deviation_topk_noalloc(kf, kr, reqs, policy, got)
        torch.cuda.synchronize()
        assert R.device_status() == 0
        assert torch.equal(got, ref)


def test_noalloc_ignores_the_callers_dev_offset():
    """dev_offset is not an input here: a C caller that leaves it at any
    value (here -1, which cb_kv_deviation_topk would reject) gets the same
    selection."""
    import ctypes as C
    kf, kr, reqs, k_total, n_total = _inputs(3)
    ref = torch.full((k_total,), -1, dtype=torch.int32, device="cuda")
    d = torch.empty(n_total, dtype=torch.float32, device="cuda")
    R.cb_kv_deviation_topk(kf, kr, reqs, L.CB_POLICY_TOKEN_TOPK, d, ref)
    arr = (L.SelectReq * len(reqs))()
    for i, r in enumerate(reqs):
        arr[i] = L.SelectReq(r["n_ctx"], r["k"], r["fresh_row0"], r["reused_row0"], -1,
                             r["idx_offset"], 0, None, None, 0, 0)
    got = torch.full((k_total,), -2, dtype=torch.int32, device="cuda")
    L.check(L.lib.cb_kv_deviation_topk_noalloc(
        C.c_void_p(kf.data_ptr()), kf.stride(0), C.c_void_p(kr.data_ptr()), kr.stride(0),
        kf.shape[1], L.CB_BF16, arr, len(reqs), L.CB_POLICY_TOKEN_TOPK,
        C.c_void_p(got.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    assert R.device_status() == 0
    assert torch.equal(got, ref)


def test_noalloc_rejects_more_than_its_limit():
    # inputs that hold every row the request names (8 bf16 = 16 bytes per
    # row), so a limit check that let the call through would read in bounds
    # and show up only as the missing error below
    n = (1 << 20) + 1
    kf = torch.zeros(n, 8, dtype=torch.bfloat16, device="cuda")
    reqs = [dict(n_ctx=n, k=1)]
    with pytest.raises(L.CBError) as e:
        R.cb_kv_deviation_topk_noalloc(kf, kf, reqs, L.CB_POLICY_TOKEN_TOPK,
                                       torch.empty(1, dtype=torch.int32, device="cuda"))
    assert e.value.status == L.CB_ERR_INVALID_ARG
    assert "1048576" in str(e.value)
