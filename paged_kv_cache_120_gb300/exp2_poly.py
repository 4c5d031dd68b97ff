"""Coefficients of the polynomial 2^f ~ p(f) on [-1/2, 1/2] that the prefill
softmax evaluates on the FMA pipe for part of its exponentials.

Method: the Remez exchange algorithm (E. Ya. Remez, 1934) for the minimax
*relative* error of a degree-n polynomial: solve for the coefficients and the
levelled error on n + 2 reference points, move the references to the extrema
of the new error curve, repeat until they settle. The kernel then computes
2^x as 2^j * p(f) with j = round(x), f = x - j (range reduction in the manner
of Cody and Waite, exact in fp32 for |x| < 2^22), inserting j into the
exponent field with one integer add.

Run ``python -m paged_kv_cache_120_gb300.exp2_poly`` to print the fp32
coefficients and the bounds that ``csrc/pa_prefill.cu`` quotes.
"""
from __future__ import annotations

import numpy as np

LO, HI = -0.5, 0.5


def remez_relative(degree: int, iters: int = 40):
    """Minimax relative-error fit of 2^f on [LO, HI]; returns (coefficients
    low order first, float64; levelled error)."""
    n = degree + 2
    # Chebyshev extrema as the first reference set
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(LO, HI, 400001)
    c = None
    for _ in range(iters):
        f = np.exp2(x)
        a = np.zeros((n, n))
        for i in range(degree + 1):
            a[:, i] = x ** i
        a[:, degree + 1] = ((-1.0) ** np.arange(n)) * f
        sol = np.linalg.solve(a, f)
        c = sol[:degree + 1]
        err = np.polyval(c[::-1], grid) / np.exp2(grid) - 1.0
        # one extremum per sign run of the error curve
        sign = np.sign(err)
        cuts = np.flatnonzero(sign[1:] != sign[:-1]) + 1
        runs = np.split(np.arange(grid.size), cuts)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) != n:
            break
        x = grid[ext]
    return c, float(np.max(np.abs(np.polyval(c[::-1], grid) / np.exp2(grid) - 1.0)))


def fp32_coefficients(degree: int) -> list:
    c, _ = remez_relative(degree)
    return [float(np.float32(v)) for v in c]


def emulate(x, coeffs) -> np.ndarray:
    """The kernel's fp32 sequence, step for step, on numpy float32 values:
    clamp below at -126 (NaN kept), j = round(x) by adding and subtracting
    1.5 * 2^23, f = x - j, Horner with fused multiply-adds (emulated in
    float64 then rounded, which is what a fused multiply-add returns for
    these magnitudes), exponent field += j."""
    x = np.asarray(x, dtype=np.float32)
    x = np.where(np.isnan(x), x, np.maximum(x, np.float32(-126.0)))
    magic = np.float32(12582912.0)
    j = (x + magic).astype(np.float32)
    t = (j - magic).astype(np.float32)
    f = (x - t).astype(np.float32)
    c = [np.float32(v) for v in coeffs]
    p = c[-1]
    for ck in reversed(c[:-1]):
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(ck)).astype(np.float32)
    bits = p.view(np.uint32).astype(np.uint64) + (j.view(np.uint32).astype(np.uint64) << np.uint64(23))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    for d in (3, 4):
        c64, e = remez_relative(d)
        c32 = fp32_coefficients(d)
        xs = np.linspace(-30.0, 8.5, 2000001, dtype=np.float32)
        got = emulate(xs, c32).astype(np.float64)
        rel = np.max(np.abs(got / np.exp2(xs.astype(np.float64)) - 1.0))
        print(f"degree {d}: levelled error {e:.3e}, fp32 sequence max rel error {rel:.3e}")
        print("   ", ", ".join(f"{v!r}f" for v in c32), " (", ", ".join(float.hex(v) for v in c32), ")")
