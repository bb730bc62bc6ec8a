"""Derive the coefficients of the FMA-pipe base-2 exponential used by the
kernel for part of the softmax probabilities.

Method (Cody and Waite's range reduction followed by a minimax polynomial,
the standard textbook construction):

    2^x = 2^n * 2^f,   n = round-to-nearest(x),   f = x - n in [-1/2, 1/2]

2^n is applied by adding n to the IEEE exponent field; 2^f is approximated
on [-1/2, 1/2] by c0 + c1 f + c2 f^2 + c3 f^3 with c0 fixed to exactly 1 (so
an input clamped to -127 returns exactly +0.0 after the exponent add, and
f = 0 returns exactly 2^n).  c1..c3 minimise the maximum RELATIVE error on
a dense grid, solved as a linear program (the minimax criterion of the
Remez method, without the exchange iteration).

Running this file prints the coefficients as float32 hex and decimal; the
CPU test ``tests/test_exp2_poly.py`` re-runs the fit and checks that the
constants compiled into ``csrc/sdpa_fwd_sm103a.cu`` match it and that the
float32 evaluation order used in the kernel keeps the relative error below
2^-12 (the probabilities are rounded to bf16 / fp16 right after, which have
2^-9 / 2^-11 relative precision).
"""
from __future__ import annotations

import numpy as np


def minimax_exp2(degree: int = 3, grid: int = 4001):
    """Minimax (relative error) polynomial for 2^f on [-1/2, 1/2] with c0 = 1.

    With c0 pinned the error vanishes at f = 0, which breaks the usual
    alternation count of the Remez exchange, so the problem is solved
    directly as the linear program it is on a dense grid:
        minimise E  subject to  |(1 + sum_i c_i f^i) / 2^f - 1| <= E."""
    from scipy.optimize import linprog

    f = np.linspace(-0.5, 0.5, grid)
    w = np.exp2(-f)
    # variables: c1..c_degree, E
    basis = np.stack([f ** i * w for i in range(1, degree + 1)], axis=1)
    rhs = 1.0 - w
    ones = np.ones((grid, 1))
    A_ub = np.vstack([np.hstack([basis, -ones]), np.hstack([-basis, -ones])])
    b_ub = np.concatenate([rhs, -rhs])
    cost = np.zeros(degree + 1)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1),
                  method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    coef = np.concatenate([[1.0], res.x[:degree]])
    return coef, float(res.x[-1])


def coefficients_f32():
    coef, _ = minimax_exp2()
    return [np.float32(c) for c in coef]


def exp2_poly_f32(x: np.ndarray, coef=None) -> np.ndarray:
    """float32 emulation of the kernel's sequence of operations."""
    c = coefficients_f32() if coef is None else [np.float32(v) for v in coef]
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)  # 1.5 * 2^23: adding it rounds to an integer
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c[3])
    p = (p * f + c[2]).astype(np.float32)  # the kernel uses fused multiply-adds;
    p = (p * f + c[1]).astype(np.float32)  # float32 products here round twice,
    p = (p * f + c[0]).astype(np.float32)  # which only loosens the bound checked
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.view(np.float32)


if __name__ == "__main__":
    coef, e = minimax_exp2()
    print(f"max relative error of the real-coefficient polynomial: {e:.3e} (2^{np.log2(e):.2f})")
    for i, c in enumerate(coefficients_f32()):
        print(f"c{i} = {float(c):.9e}f  /* 0x{np.float32(c).view(np.uint32):08x} */")
