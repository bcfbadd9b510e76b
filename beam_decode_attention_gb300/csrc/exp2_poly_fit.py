"""Derives the cubic used for part of the exp2 evaluations in gr_ctx_tc.cu.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]; 2^f is
approximated by a cubic whose coefficients minimise the maximum relative
error on that interval (iteratively reweighted least squares on a dense
grid, the weights growing where the error is large).  The result (max
relative error about 7.5e-5) is far below the bf16 rounding the
probabilities undergo afterwards (2^-9).  Run: python exp2_poly_fit.py
"""
import numpy as np

f = np.linspace(-0.5, 0.5, 20001)
y = np.exp2(f)
V = np.vander(f, 4, increasing=True)
w = 1.0 / y
for it in range(200):
    A = V * w[:, None]
    b = y * w
    c, *_ = np.linalg.lstsq(A, b, rcond=None)
    err = (V @ c - y) / y
    w = w * (1 + 50 * np.abs(err) / np.abs(err).max()) ** 0.5
    w /= w.mean()
c32 = c.astype(np.float32)
err32 = (np.polyval(c32[::-1].astype(np.float64), f) - y) / y
print("coeffs", [float(x) for x in c32], "max rel err", np.abs(err32).max())
