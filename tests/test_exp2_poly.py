"""The attention kernel computes part of its exponentials on the FMA pipe
(exp2_poly in k_attn_tc.cu): x = n + f with n = round(x) taken from the
1.5 * 2^23 shift, 2^f from a cubic, n added to the exponent field.  This
test re-derives the cubic (least squares on the relative error at
Chebyshev nodes of [-1/2, 1/2]), checks the constants in the source, and
replays the kernel's float32 arithmetic against 2^x.  No GPU."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "rag_kv_cache_layer_gb300", "csrc", "k_attn_tc.cu")


def _kernel_coeffs():
    text = open(SRC).read()
    return [float(re.search(rf"kExpC{i} = ([0-9.]+)f", text).group(1)) for i in range(4)]


def _fit():
    n = 8192
    f = 0.5 * np.cos(np.pi * (np.arange(n) + 0.5) / n)
    y = 2.0 ** f
    A = np.stack([f ** k for k in range(4)], 1) / y[:, None]
    c, *_ = np.linalg.lstsq(A, np.ones(n), rcond=None)
    return c


def _exp2_poly(x, c):
    """The kernel's steps in float32 (fmaf emulated in float64 and rounded)."""
    c = np.float32(c)
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(f32)
    f = (x - (t - f32(12582912.0))).astype(f32)
    p = f32(np.float64(c[3]) * f + c[2])
    p = f32(np.float64(p) * f + c[1])
    p = f32(np.float64(p) * f + c[0])
    bits = p.view(np.int32) + (t.view(np.int32) << np.int32(23))
    return bits.view(np.float32)


def test_coefficients_are_the_fit():
    assert np.allclose(_kernel_coeffs(), _fit(), rtol=0, atol=5e-7)


def test_relative_error_below_bf16_resolution():
    c = np.array(_kernel_coeffs())
    x = np.concatenate([np.linspace(-125.0, 8.0, 400001), np.arange(-125, 9, dtype=np.float64)])
    got = _exp2_poly(x, c).astype(np.float64)
    rel = np.abs(got / 2.0 ** x.astype(np.float32).astype(np.float64) - 1)
    assert rel.max() < 1e-4          # bf16 rounding of p is 2^-9 = 2e-3


def test_tiny_arguments_flush_to_negligible_values():
    c = np.array(_kernel_coeffs())
    got = _exp2_poly(np.array([-126.0, -200.0, -1e30]), c).astype(np.float64)
    assert np.all(np.isfinite(got)) and np.all(got >= 0) and np.all(got < 2.0 ** -120)
