"""Print the coefficients of exp2_poly.h: minimax fits of 2^f on [-1/2, 1/2].

p(f) = 1 + c1 f + ... + cd f^d, with p(0) = 1 held exactly, minimising the
largest relative error |p(f) / 2^f - 1| over a dense grid of f, posed as a
linear program (minimise t subject to -t <= (p(f_i) - 2^f_i) / 2^f_i <= t).
The coefficients are then rounded to fp32 and the fp32 Horner evaluation is
re-measured on the grid.

    python exact_long_sequence_gb300/csrc/fit_exp2_poly.py
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree: int, points: int = 20001):
    f = np.linspace(-0.5, 0.5, points)
    e = np.exp2(f)
    a = np.stack([f ** k / e for k in range(1, degree + 1)], 1)  # (p - e) / e = 1/e - 1 + a c
    b = 1.0 - 1.0 / e
    ones = np.ones((points, 1))
    a_ub = np.vstack([np.hstack([a, -ones]), np.hstack([-a, -ones])])
    b_ub = np.concatenate([b, -b])
    cost = np.zeros(degree + 1)
    cost[-1] = 1.0
    r = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * degree + [(0, None)], method="highs")
    return r.x[:degree], r.x[-1]


def fp32_relative_error(c32):
    f = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    acc = np.full_like(f, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        acc = (acc.astype(np.float64) * f + np.float64(c32[k])).astype(np.float32)  # one rounding, as fmaf
    p = (acc.astype(np.float64) * f + 1.0).astype(np.float32)
    return float(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0).max())


if __name__ == "__main__":
    for degree in (3, 4, 5):
        c, t = fit(degree)
        c32 = c.astype(np.float32)
        print(f"degree {degree}: minimax {t:.3e}, fp32 {fp32_relative_error(c32):.3e}: "
              + ", ".join(float(x).hex() for x in c32))
