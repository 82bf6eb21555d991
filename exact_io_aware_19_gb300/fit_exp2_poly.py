"""Fit the polynomial the attention kernel uses for part of its exp2 evaluations.

The kernel evaluates 2^x as 2^j · p(f), with j = round(x) and f = x - j in
[-1/2, 1/2] (Cody–Waite style range reduction; j is added to the exponent
field). p is the degree-3 polynomial that minimises the maximum relative error
|p(f) / 2^f - 1| on [-1/2, 1/2]. It is found here as a linear program on a dense
grid (minimise t subject to |p(f_i) - 2^f_i| <= t · 2^f_i), rounded to fp32, and its
error is re-measured with fp32 Horner evaluation.

    python -m exact_io_aware_19_gb300.fit_exp2_poly      # rewrites csrc/exp2_poly.h

Why a polynomial at all: on GB300 the MUFU ex2 unit issues 32 results per clock
per SM, exactly the rate the d = 64 tensor-core work of a softmax block needs;
moving a fraction of the exponentials to the FMA pipes leaves the MUFU slack.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.optimize import linprog

DEGREE = 3
HEADER = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "exp2_poly.h")


def fit(degree: int = DEGREE, n: int = 4001):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)  # columns f^0 .. f^degree
    # variables: c_0..c_degree, t ; minimise t
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    A = np.vstack([np.hstack([V, -y[:, None]]), np.hstack([-V, -y[:, None]])])
    b = np.concatenate([y, -y])
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * (degree + 1) + [(0, None)],
                  method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:-1], res.x[-1]


def fp32_error(coef, n: int = 200001) -> float:
    """Max relative error of fp32 Horner evaluation of p on [-1/2, 1/2]."""
    c = np.asarray(coef, dtype=np.float32)
    f = np.linspace(-0.5, 0.5, n).astype(np.float32)
    p = np.full_like(f, c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = (p * f + c[k]).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


def main():
    coef, t = fit()
    c32 = [float(np.float32(x)) for x in coef]
    err = fp32_error(c32)
    lines = [
        "// exp2_poly.h — written by exact_io_aware_19_gb300/fit_exp2_poly.py; do not edit.",
        f"// Degree-{DEGREE} minimax fit of 2^f on [-1/2, 1/2] (relative error), fp32 coefficients.",
        f"// LP optimum {t:.3e}; measured with fp32 Horner evaluation: {err:.3e}.",
        "#pragma once",
        "",
        "namespace ex19 {",
        f"constexpr float kExp2PolyMaxRelErr = {err:.3e}f;",
    ]
    for k, c in enumerate(c32):
        lines.append(f"constexpr float kExp2C{k} = {c!r}f;")
    lines += ["}  // namespace ex19", ""]
    with open(HEADER, "w") as fh:
        fh.write("\n".join(lines))
    print("\n".join(lines))


if __name__ == "__main__":
    main()
