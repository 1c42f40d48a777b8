"""Fits the polynomial the scan kernels use for log1p(w), w in [0, 1].

log1p(w) is written as w * Q(w) with Q of degree 8. Q is fitted to
log1p(w) / w by weighted least squares on 4000 Chebyshev nodes of [0, 1],
reweighted by Lawson's iteration towards the minimax (equal-ripple) solution
of the relative error. The coefficients are rounded to float32 and the
relative error of w * Q(w), evaluated by Horner's rule in float32 arithmetic
on a 200000-point grid, is printed (2.3e-7).

Run: python selective_state_space_138_b300/csrc/fit_log1p.py
"""
import numpy as np

DEG = 8


def fit(deg=DEG, nodes_n=4000, iters=60):
    k = np.arange(nodes_n)
    w = 0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / nodes_n)
    f = np.log1p(w) / w
    V = np.vander(w, deg + 1, increasing=True)
    inv = 1.0 / f
    weights = np.ones_like(w)
    coef = None
    for _ in range(iters):
        sw = inv * np.sqrt(weights)
        coef, *_ = np.linalg.lstsq(V * sw[:, None], f * sw, rcond=None)
        err = np.abs((V @ coef - f) / f)
        weights = weights * err
        weights /= weights.sum()
    return coef.astype(np.float32)


def max_rel_error_float32(c32):
    w = np.linspace(0, 1, 200001, dtype=np.float32)[1:]
    q = np.full_like(w, c32[-1])
    for c in c32[-2::-1]:
        q = (q * w + c).astype(np.float32)
    r = (w * q).astype(np.float32)
    ref = np.log1p(w.astype(np.float64))
    return float(np.max(np.abs(r - ref) / ref))


if __name__ == "__main__":
    c = fit()
    print("coefficients (w^0 .. w^%d):" % DEG)
    for v in c:
        print("  %.9ef" % v)
    print("max relative error (float32 Horner): %.2e" % max_rel_error_float32(c))
