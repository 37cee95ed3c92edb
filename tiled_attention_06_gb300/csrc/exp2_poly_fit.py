"""Coefficients of the polynomial that the prefill softmax uses for part of its 2^f.

The kernel splits x = r + f with r = rint(x) and f in [-1/2, 1/2] (Cody-Waite style range
reduction with a single constant, exact because the rounding is done by adding and
subtracting 1.5 * 2^23), approximates 2^f by a polynomial and puts r into the exponent
field. The polynomial is the discrete minimax fit in RELATIVE error on a dense grid of
[-1/2, 1/2]: minimise e subject to |p(f_i) / 2^f_i - 1| <= e, a linear program in
(c_0..c_n, e). Run this file to print the coefficients (float32) and the fit's error.
"""
import sys

import numpy as np
from scipy.optimize import linprog


def fit(degree: int = 3, n: int = 4001):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True) / y[:, None]  # p(f)/2^f, linear in c
    # variables (c_0..c_n, e); minimise e;  V c - e <= 1  and  -V c - e <= -1
    A = np.vstack([np.hstack([V, -np.ones((n, 1))]), np.hstack([-V, -np.ones((n, 1))])])
    b = np.concatenate([np.ones(n), -np.ones(n)])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * (degree + 2), method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:-1].astype(np.float32), float(res.x[-1])


def rel_error(c, n: int = 200001) -> float:
    f = np.linspace(-0.5, 0.5, n)
    p = np.zeros_like(f)
    for ck in np.asarray(c, dtype=np.float64)[::-1]:
        p = p * f + ck
    return float(np.max(np.abs(p / np.exp2(f) - 1.0)))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c, e = fit(deg)
    for k, ck in enumerate(c):
        print(f"c{k} = {float(ck):.9e}f")
    print(f"fit error {e:.3e}; with float32 coefficients {rel_error(c):.3e}")
