"""Coefficients of the polynomial 2^f ~ c0 + c1 f + c2 f^2 + c3 f^3 on
f in [-1/2, 1/2] used by the forward kernel's FMA-pipe exp2.

Method: range reduction 2^x = 2^n * 2^f with n = round(x) (Cody and Waite,
"Software Manual for the Elementary Functions", 1980), and a polynomial for
2^f fitted by least squares on Chebyshev nodes, weighted for relative error
(a near-minimax fit), in fp64, then rounded to f32.  c0 is pinned to 1 so
that 2^0 is exact.  Run:  python exp2_poly_fit.py  -> prints the f32
coefficients and the worst relative error of the f32 Horner evaluation on a
dense grid.
"""
import numpy as np


def fit(degree: int = 3, nodes: int = 4096):
    k = np.arange(nodes)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / nodes)          # Chebyshev nodes on [-1/2, 1/2]
    target = np.exp2(f)
    # c0 = 1 fixed: fit (2^f - 1) / f ~ c1 + c2 f + c3 f^2, relative weights 1/2^f
    w = 1.0 / target
    A = np.stack([f ** (i + 1) for i in range(degree)], axis=1) * w[:, None]
    b = (target - 1.0) * w
    c = np.linalg.lstsq(A, b, rcond=None)[0]
    return np.concatenate([[1.0], c])


def horner_f32(c, f):
    c = c.astype(np.float32)
    f = f.astype(np.float32)
    p = np.full_like(f, c[-1])
    for ci in c[-2::-1]:
        p = (p * f + ci).astype(np.float32)
    return p


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs(horner_f32(c, f).astype(np.float64) / np.exp2(f) - 1.0).max()
    print("c =", ", ".join(f"{np.float32(x).item()!r}f" for x in c))
    print("max relative error (f32 Horner) =", rel)
