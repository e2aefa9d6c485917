"""Fit the polynomial behind the FMA-pipe exp2 of the forward kernel.

Method (published): Cody & Waite range reduction, x = n + f with n the
nearest integer and f in [-1/2, 1/2], so 2^x = 2^n * 2^f; 2^f is replaced by
the degree-3 polynomial minimising the maximum *relative* error on
[-1/2, 1/2], found with the Remez exchange algorithm (equioscillation at 5
points). Coefficients are rounded to float32. The kernel evaluates the
polynomial in Horner form with fused multiply-adds and adds n to the
exponent field.

Run: python fit_exp2_poly.py  -> prints the coefficients and the error.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def remez(degree: int = DEGREE, iters: int = 30):
    """Minimax relative-error fit of 2^f on [LO, HI]: returns float64 coeffs c0..cd."""
    m = degree + 2
    # start from Chebyshev extrema
    k = np.arange(m)
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * -np.cos(np.pi * k / (m - 1))
    grid = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        # solve  sum c_i x^i - 2^x = (-1)^j E 2^x   (relative error equioscillates)
        A = np.zeros((m, m))
        for j in range(m):
            A[j, :degree + 1] = x[j] ** np.arange(degree + 1)
            A[j, degree + 1] = -((-1) ** j) * 2.0 ** x[j]
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:degree + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: extrema of the error between sign changes
        sign_changes = np.nonzero(np.diff(np.sign(err)))[0]
        bounds = [0, *list(sign_changes + 1), len(grid)]
        ext = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            seg = np.abs(err[a:b])
            ext.append(a + int(np.argmax(seg)))
        if len(ext) < m:
            break
        # keep m alternating extrema with the largest magnitudes
        while len(ext) > m:
            drop = 0 if abs(err[ext[0]]) < abs(err[ext[-1]]) else len(ext) - 1
            ext.pop(drop)
        x = grid[ext]
    return c


def f32_coeffs(c):
    return [float(np.float32(v)) for v in c]


def emulate(x: np.ndarray, coeffs) -> np.ndarray:
    """float32 emulation of the kernel's sequence of operations."""
    x = np.maximum(np.asarray(x, np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)              # 1.5 * 2^23: rounds to an integer
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    c = [np.float32(v) for v in coeffs]
    p = c[3]
    p = (p * f + c[2]).astype(np.float32)       # fma rounding differences are below 1 ulp
    p = (p * f + c[1]).astype(np.float32)
    p = (p * f + c[0]).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.astype(np.int32).view(np.float32)


def main():
    c = f32_coeffs(remez())
    xs = np.linspace(-125.0, 8.0, 2000001, dtype=np.float32)
    rel = np.abs(emulate(xs, c).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1.0)
    print("coefficients c0..c3 (float32):")
    for v in c:
        print(f"  {v!r}  ({np.float32(v).view(np.uint32):#010x})")
    print(f"max relative error on [-125, 8]: {rel.max():.3e}")


if __name__ == "__main__":
    main()
