"""Coefficients of the softplus polynomial used by the scan kernels.

softplus(x) = max(x, 0) + log1p(e),  e = exp(-|x|) in (0, 1].
log1p(e) is evaluated as e * P(e), where P is a degree-8 polynomial fitted
here by least squares to log1p(e)/e at 4000 Chebyshev nodes of [0, 1]
(fp64), then rounded to fp32.  Evaluated in fp32 by Horner's rule, the
relative error of e * P(e) against log1p(e) is below 2e-7 on [0, 1].

    python gen_log1p_poly.py      # prints the coefficients and the error bound
"""
import numpy as np

DEG = 8


def coefficients(deg=DEG):
    xs = (np.cos(np.pi * (np.arange(4000) + 0.5) / 4000) + 1.0) / 2.0
    f = np.log1p(xs) / xs
    V = np.vander(xs, deg + 1, increasing=True)
    c, *_ = np.linalg.lstsq(V, f, rcond=None)
    return c.astype(np.float32)


def max_rel_error(c):
    e = np.linspace(0.0, 1.0, 400001).astype(np.float32)
    p = np.full_like(e, c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = (p * e + c[k]).astype(np.float32)
    got = (e * p).astype(np.float64)
    ref = np.log1p(e.astype(np.float64))
    m = ref > 0
    return float(np.max(np.abs(got[m] - ref[m]) / ref[m]))


if __name__ == "__main__":
    c = coefficients()
    for k, v in enumerate(c):
        print(f"c{k} = {float(v)!r}f")
    print("max relative error of e*P(e):", max_rel_error(c))
