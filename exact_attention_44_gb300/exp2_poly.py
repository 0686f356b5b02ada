"""Coefficients of the polynomial the softmax kernels use for part of their
base-2 exponentials (the rest go through the MUFU unit's ex2).

    python -m exact_attention_44_gb300.exp2_poly        # print them as C++

Method (both published, stated here from their definitions):

* Cody-Waite range reduction, base 2: for x >= -126, n = round(x) and
  f = x - n in [-1/2, 1/2] (exact in fp32 for |x| < 2^22); 2^x = 2^n * 2^f,
  and 2^n is applied by adding n to the exponent field of 2^f.
* A minimax polynomial p(f) ~ 2^f on [-1/2, 1/2], minimising the maximum
  RELATIVE error |p(f) / 2^f - 1|, found with the Remez exchange algorithm:
  on degree + 2 reference points solve p(t_i) - (-1)^i E 2^t_i = 2^t_i for
  the coefficients and the levelled error E, move the references to the
  extrema of the error function, repeat until they stop moving.

The kernel evaluates p in Horner form with fp32 fused multiply-adds; the
coefficients below are the Remez solution rounded to fp32.  The tests check
the stored constants against this script and the fp32 evaluation against
numpy's exp2 over the kernel's input range.
"""
from __future__ import annotations

import numpy as np

DEGREE = 4
LO, HI = -0.5, 0.5


def _error(c, t):
    return np.polyval(c[::-1], t) / np.exp2(t) - 1.0


def remez(degree: int = DEGREE, iters: int = 60, grid: int = 200001):
    """Minimax-relative-error coefficients c[0..degree] (lowest order first) and the levelled error."""
    n = degree + 2
    k = np.arange(n)
    t = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * (n - 1 - k) / (n - 1))  # Chebyshev extrema
    xs = np.linspace(LO, HI, grid)
    E = 0.0
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :degree + 1] = t[i] ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1) ** i) * np.exp2(t[i])
        sol = np.linalg.solve(A, np.exp2(t))
        c, E = sol[:degree + 1], sol[degree + 1]
        e = _error(c, xs)
        # new references: the extremum of the error in each run of one sign
        sign = np.sign(e)
        sign[sign == 0] = 1
        cuts = np.flatnonzero(np.diff(sign)) + 1
        runs = np.split(np.arange(grid), cuts)
        ext = np.array([r[np.argmax(np.abs(e[r]))] for r in runs])
        if len(ext) > n:  # keep the n consecutive extrema with the largest smallest magnitude
            best = max(range(len(ext) - n + 1), key=lambda s: np.min(np.abs(e[ext[s:s + n]])))
            ext = ext[best:best + n]
        if len(ext) < n:
            break
        t_new = xs[ext]
        if np.max(np.abs(t_new - t)) < 1e-12:
            t = t_new
            break
        t = t_new
    return c, abs(E)


def coefficients_f32(degree: int = DEGREE):
    c, _ = remez(degree)
    return [float(np.float32(x)) for x in c]


def evaluate_f32(x: np.ndarray, coeffs=None) -> np.ndarray:
    """The kernel's computation, step by step in fp32 (numpy's float32 rounds each operation;
    the kernel's fused multiply-adds round once, which is at least as accurate)."""
    coeffs = coefficients_f32() if coeffs is None else coeffs
    f32 = np.float32
    x = np.maximum(np.asarray(x, dtype=np.float32), f32(-126.0))
    magic = f32(12582912.0)  # 1.5 * 2^23: x + magic rounds x to an integer in the low mantissa bits
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.full_like(f, f32(coeffs[-1]))
    for ck in coeffs[-2::-1]:
        p = (p * f + f32(ck)).astype(np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def as_cpp(coeffs=None) -> str:
    coeffs = coefficients_f32() if coeffs is None else coeffs
    body = ", ".join(f"{float(v).hex()}f" for v in coeffs)
    return f"constexpr float EXP2_POLY[{len(coeffs)}] = {{{body}}};"


if __name__ == "__main__":
    c, err = remez()
    print(f"// degree {DEGREE} minimax of 2^f on [-1/2, 1/2], max relative error {err:.3e}")
    print(as_cpp())
