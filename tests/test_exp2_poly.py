"""The FMA-pipe 2^x used for part of the prefill softmax exponentials: the
same float32 steps as the kernel (range reduction by x + 1.5*2^23, degree-4
polynomial for 2^f, exponent added to the bits) against numpy's exp2."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "paged_kv_cache_316_gb300", "csrc", "prefill.cu")


def kernel_coefficients():
    body = open(SRC).read()
    fn = body[body.index("float exp2_fma(float x)"):]
    fn = fn[:fn.index("return x < -126.f")]
    return [np.float32(float(v)) for v in re.findall(r"([0-9.]+e[-+][0-9]+)f", fn)]


def exp2_fma(x):
    x = np.asarray(x, np.float32)
    c4, c3, c2, c1 = kernel_coefficients()
    xc = np.maximum(x, np.float32(-126))
    t = (xc + np.float32(12582912.0)).astype(np.float32)
    f = (xc - (t - np.float32(12582912.0))).astype(np.float32)
    q = (c4 * f + c3).astype(np.float32)
    q = (q * f + c2).astype(np.float32)
    q = (q * f + c1).astype(np.float32)
    q = (q * f + np.float32(1.0)).astype(np.float32)
    bits = q.view(np.int32) + (t.view(np.int32) << 23)
    r = bits.view(np.float32)
    return np.where(x < -126, np.float32(0), r)


def test_relative_error_over_softmax_range():
    x = np.linspace(-125.5, 8.0, 2_000_001, dtype=np.float64).astype(np.float32)
    got = exp2_fma(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / ref - 1.0)) < 1e-5


def test_masked_and_integer_inputs():
    assert exp2_fma(np.float32(-np.inf)) == 0
    assert exp2_fma(np.float32(-200)) == 0
    for n in range(-20, 9):
        assert abs(float(exp2_fma(np.float32(n))) / 2.0 ** n - 1) < 1e-6
