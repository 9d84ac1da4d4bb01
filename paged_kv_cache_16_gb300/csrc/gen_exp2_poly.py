"""Coefficients of the polynomial 2^f ~= c0 + c1 f + c2 f^2 + c3 f^3 on [-1/2, 1/2].

Used by the softmax of the tensor-core tile to evaluate part of its
exponentials on the FMA pipe instead of the special-function unit.  The fit
minimises the maximum relative error (Lawson's iteratively reweighted least
squares on a dense grid, which converges to the minimax fit).  Prints the
coefficients as float32 literals and the fit's relative error bound.

    python paged_kv_cache_16_gb300/csrc/gen_exp2_poly.py
"""
import numpy as np

DEGREE = 3


def fit(degree=DEGREE, n=20001, iters=200):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True) / y[:, None]   # relative error system
    w = np.ones(n) / n
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V * sw[:, None], sw, rcond=None)
        r = np.abs(V @ c - 1.0)
        w = w * r
        w /= w.sum()
    c32 = c.astype(np.float32)
    # error of the float32 coefficients evaluated in float64
    rel = np.abs(np.polyval(c32[::-1].astype(np.float64), f) / y - 1.0).max()
    return c32, rel


if __name__ == "__main__":
    c, rel = fit()
    for i, v in enumerate(c):
        print(f"c{i} = {float(v)!r}f")
    print(f"max relative error on [-0.5, 0.5]: {rel:.3e}")
