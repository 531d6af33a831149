"""Coefficients of the cubic that the prefill kernel uses for part of its
exp2 evaluations (on the FMA pipe, to relieve the MUFU unit).

2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2], and 2^f is
approximated by the degree-3 polynomial minimising the maximum relative
error on [-1/2, 1/2], found by the Remez exchange algorithm starting from
Chebyshev points.  Run this module to print the coefficients and the error
bound; tests check that the kernel's constants match.

    python -m paged_kv_cache_124_gb300.exp2_poly_fit
"""
import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _relerr(c, x):
    return np.polyval(c[::-1], x) / 2.0 ** x - 1.0


def fit(degree=DEGREE, iters=20, samples=200001):
    grid = np.linspace(LO, HI, samples)
    n = degree + 2
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    c = None
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i at the reference points
        A = np.hstack([np.vander(x, degree + 1, increasing=True), (-(-1.0) ** np.arange(n) * 2.0 ** x)[:, None]])
        c = np.linalg.solve(A, 2.0 ** x)[:-1]
        e = _relerr(c, grid)
        ext = [0] + [i for i in range(1, samples - 1) if (e[i] - e[i - 1]) * (e[i + 1] - e[i]) <= 0] + [samples - 1]
        ext = np.array(ext)
        x = np.sort(grid[ext[np.argsort(-np.abs(e[ext]))][:n]])
    return c, float(np.abs(_relerr(c, grid)).max())


def fp32_max_relerr(c, samples=200001):
    """Maximum relative error of the cubic evaluated in float32 by Horner's rule."""
    cf = np.asarray(c, dtype=np.float32)
    f = np.linspace(LO, HI, samples).astype(np.float32)
    p = ((cf[3] * f + cf[2]) * f + cf[1]) * f + cf[0]
    return float(np.abs(p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1).max())


if __name__ == "__main__":
    c, err = fit()
    print("coefficients c0..c3:", ", ".join("%.9e" % v for v in c))
    print("max relative error %.3e (float32 Horner %.3e)" % (err, fp32_max_relerr(c)))
