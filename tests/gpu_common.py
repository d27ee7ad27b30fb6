"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

import workload as W

F32_ATOL = 1e-4          # max-abs bound for float32 outputs
BF16_RMS = 2e-2          # RMS-relative bound for bf16 outputs


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rms_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.sqrt(np.mean((got - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30))


def assert_close(got, ref, dtype):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if dtype == torch.float32:
        err = float(np.max(np.abs(got - ref))) if got.size else 0.0
        assert err <= F32_ATOL, f"max abs err {err}"
    else:
        r = rms_rel(got, ref)
        assert r <= BF16_RMS, f"rms rel err {r}"


def bf16_values(a):
    """Values exactly representable in bf16 (as float32)."""
    return W.round_to_bf16(np.asarray(a, np.float32))


def ties_ok(sel_gpu, sel_ref, d_ref, k, rel=1e-3):
    """Selected sets agree except for positions whose reference deviation
    ties the k-th largest within ``rel`` (relative).  Deviations below 1e-12
    of the largest are zero up to float64 rounding -- the first chunk's are
    exactly zero in exact arithmetic ("Request Order Matters" §2.2: its
    prefix is unchanged) -- so they tie with each other and with a zero k-th
    value."""
    if k == 0:
        return len(sel_gpu) == 0
    d_ref = np.asarray(d_ref, np.float64)
    zero = 1e-12 * float(np.max(np.abs(d_ref))) if d_ref.size else 0.0
    kth = np.sort(d_ref)[::-1][k - 1]
    diff = set(map(int, sel_gpu)) ^ set(map(int, sel_ref))
    return all(abs(d_ref[i] - kth) <= max(rel * abs(kth), zero, 1e-300) for i in diff)
