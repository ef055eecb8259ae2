"""Derives the polynomial that the scan kernels use for log1p(v), v in [0, 1].

softplus(x) = max(x, 0) + log1p(exp(-|x|)) needs log1p on (0, 1]. The MUFU
log2 has an absolute error near 1e-7, which is a large RELATIVE error when
softplus is small (delta around 1e-3 is common), so the kernels evaluate
log1p(v) = v * q(v) with q a degree-7 polynomial fitted here: a weighted
least-squares fit of log1p(v)/v on Chebyshev nodes of [0, 1] (close to the
minimax fit), coefficients rounded to fp32. Run this file to print the
coefficients and the fit's error bound (relative to log1p, in float64).
"""
import numpy as np

DEG = 7


def fit(deg=DEG, nodes=4000):
    k = np.arange(nodes)
    v = 0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / nodes)       # Chebyshev nodes on [0, 1]
    target = np.where(v > 0, np.log1p(v) / np.where(v > 0, v, 1), 1.0)
    V = np.vander(v, deg + 1, increasing=True)
    coef, *_ = np.linalg.lstsq(V, target, rcond=None)
    return coef.astype(np.float32)


def max_rel_error(coef, samples=200001):
    v = np.linspace(1e-9, 1.0, samples)
    q = np.polynomial.polynomial.polyval(v, coef.astype(np.float64))
    return float(np.max(np.abs(v * q - np.log1p(v)) / np.log1p(v)))


if __name__ == "__main__":
    c = fit()
    print("coefficients (increasing powers):")
    for i, x in enumerate(c):
        print(f"  c{i} = {float(x)!r}f")
    print("max relative error of v*q(v) vs log1p(v) on (0,1]:", max_rel_error(c))
