"""The FMA-pipe exponential used by the softmax of the tensor-core tile.

Its steps are replayed here in float32 numpy with the coefficients read
from the CUDA source, and checked against exp2 in float64 over the whole
input range the softmax feeds it (x <= 8; below -120 the result only has to
be negligible).  The coefficients must also match a fresh run of the fit.
"""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = os.path.join(ROOT, "paged_kv_cache_16_gb300", "csrc", "dev.cuh")
sys.path.insert(0, os.path.join(ROOT, "paged_kv_cache_16_gb300", "csrc"))


def source_coefficients():
    text = open(DEV, encoding="utf-8").read()
    body = text[text.index("float ex2_fma(float x)"):]
    body = body[:body.index("}")]
    c3 = float(re.search(r"float p = ([0-9.e-]+)f;", body).group(1))
    rest = [float(v) for v in re.findall(r"p = fmaf\(p, f, ([0-9.e-]+)f\);", body)]
    return [rest[2], rest[1], rest[0], c3]          # c0, c1, c2, c3


def fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def ex2_fma(x, coef):
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-120.0))
    k = f32(12582912.0)
    y = (x + k).astype(f32)
    f = (x - (y - k)).astype(f32)
    p = np.full_like(f, f32(coef[3]))
    for c in (coef[2], coef[1], coef[0]):
        p = fma32(p, f, np.full_like(f, f32(c)))
    bits = p.view(np.int32).astype(np.int64) + (y.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_bound():
    coef = source_coefficients()
    x = np.concatenate([np.linspace(-120.0, 8.0, 2_000_001), np.arange(-120, 9, dtype=np.float64)])
    got = ex2_fma(x.astype(np.float32), coef).astype(np.float64)
    want = np.exp2(x.astype(np.float32).astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1.0e-4, rel.max()      # fit error 7.5e-5 plus float32 rounding


def test_underflow_is_negligible():
    coef = source_coefficients()
    got = ex2_fma(np.array([-1e4, -500.0, -121.0, -np.inf], dtype=np.float32), coef)
    assert np.all(got >= 0) and np.all(got < 2.0 ** -119)


def test_coefficients_match_the_fit():
    import gen_exp2_poly
    c, rel = gen_exp2_poly.fit()
    assert np.allclose(np.asarray(source_coefficients(), np.float32), c, rtol=0, atol=2e-7)
    assert rel < 8e-5
