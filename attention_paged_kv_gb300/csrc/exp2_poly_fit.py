"""Derive the cubic that prefill.cu's exp2_fma2 uses for 2^f on [-1/2, 1/2].

Iterated reweighted least squares (Lawson's algorithm) on the relative error
over Chebyshev-spaced points converges to the minimax fit; the coefficients
are then rounded to float32 and the relative error of the float32 Horner
evaluation is reported.  Run: python exp2_poly_fit.py
"""
import numpy as np


def fit(degree: int = 3, iters: int = 200) -> np.ndarray:
    f = np.cos(np.linspace(0.0, np.pi, 4001)) * 0.5
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]
    w = np.ones_like(f)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(A * np.sqrt(w)[:, None], np.sqrt(w), rcond=None)
        e = np.abs(A @ c - 1.0)
        w = w * (e / e.max() + 1e-12)
        w /= w.sum()
    return c.astype(np.float32)


def max_rel_error(c32: np.ndarray, n: int = 200001) -> float:
    f = np.linspace(-0.5, 0.5, n).astype(np.float32)
    p = np.full_like(f, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p * f + c32[k]).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    c = fit()
    print("coefficients c0..c3:", [repr(float(x)) for x in c])
    print("max relative error:", max_rel_error(c))
