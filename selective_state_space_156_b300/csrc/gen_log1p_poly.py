"""Generates the degree-8 polynomial P with log1p(e) ~= e * P(e) on e in [0, 1] used by the
kernels' softplus (ssm_device.cuh).  Least squares in the Chebyshev basis on 4000 Chebyshev nodes,
converted to monomial coefficients and rounded to fp32; prints the coefficients and the maximum
relative error of the fp32 Horner evaluation on a dense grid.  Run: python gen_log1p_poly.py"""
import numpy as np
from numpy.polynomial import chebyshev as C

DEG = 8


def coefficients(deg=DEG):
    e = 0.5 + 0.5 * np.cos(np.pi * (np.arange(4000) + 0.5) / 4000)
    f = np.log1p(e) / e
    c = C.chebfit(2 * e - 1, f, deg)
    p = np.polynomial.Polynomial(C.cheb2poly(c))
    return p(np.polynomial.Polynomial([-1.0, 2.0])).coef.astype(np.float32)


def max_rel_error(co):
    e = np.linspace(0, 1, 400001).astype(np.float32)[1:]
    acc = np.full_like(e, co[-1])
    for c in co[-2::-1]:
        acc = (acc * e + np.float32(c)).astype(np.float32)
    val = (acc * e).astype(np.float32).astype(np.float64)
    ref = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(val - ref) / ref))


if __name__ == "__main__":
    co = coefficients()
    for i, c in enumerate(co):
        print(f"  c{i} = {float(c)!r}f")
    print("max relative error (fp32 Horner):", max_rel_error(co))
