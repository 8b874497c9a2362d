"""Coefficients of the polynomial exp2 that the kernels evaluate on the FMA pipe.

    python -m exact_attention_48_gb300.exp2_fit [--degree 5]

2^x is split exactly as 2^n * 2^f with n = round(x) and f = x - n in
[-1/2, 1/2] (for fp32 x the subtraction is exact); 2^n goes into the
exponent field with an integer add, and 2^f is a polynomial p(f) of low
degree.  This script computes p as the minimax approximation of 2^f in the
RELATIVE error on [-1/2, 1/2] with the Remez exchange algorithm (equioscillation
of e(f) = p(f) 2^-f - 1 at degree + 2 points), rounds the coefficients to
fp32, and reports the relative error of the fp32 evaluation (Horner with
fused multiply-adds, emulated) over a dense grid.  The printed table is what
csrc/exp2_poly.cuh holds.  Everything here is plain numpy in float64.
"""
from __future__ import annotations

import argparse

import numpy as np


def remez_exp2(degree: int, iters: int = 60):
    """Minimax p of the given degree for 2^f on [-1/2, 1/2], relative error."""
    n = degree
    # initial reference: Chebyshev extrema mapped to [-1/2, 1/2]
    k = np.arange(n + 2)
    ref = 0.5 * np.cos(np.pi * k / (n + 1))[::-1]
    grid = np.linspace(-0.5, 0.5, 200001)
    coef = None
    for _ in range(iters):
        # solve p(x_i) - 2^x_i (-1)^i E 2^x_i = 2^x_i  (relative error E)
        A = np.zeros((n + 2, n + 2))
        for i, x in enumerate(ref):
            A[i, : n + 1] = x ** np.arange(n + 1)
            A[i, n + 1] = (-1) ** i * 2.0 ** x
        sol = np.linalg.solve(A, 2.0 ** ref)
        coef = sol[: n + 1]
        err = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: the extrema of err on each sign-alternating run
        sign = np.sign(err)
        idx = []
        start = 0
        for j in range(1, len(grid) + 1):
            if j == len(grid) or sign[j] != sign[start]:
                seg = np.arange(start, j)
                idx.append(seg[np.argmax(np.abs(err[seg]))])
                start = j
        idx = np.array(idx)
        if len(idx) < n + 2:
            break
        # keep n + 2 alternating extrema with the largest |err|
        while len(idx) > n + 2:
            if abs(err[idx[0]]) < abs(err[idx[-1]]):
                idx = idx[1:]
            else:
                idx = idx[:-1]
        new_ref = grid[idx]
        if np.allclose(new_ref, ref, atol=1e-12):
            ref = new_ref
            break
        ref = new_ref
    return coef


def fp32_fma(a, b, c):
    """fp32 fused multiply-add, emulated: the product of two fp32 values is
    exact in float64, then one rounding of the sum to fp32 (a double
    rounding of the sum only at exact ties, which the grid below does not
    hit)."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def eval_fp32(coef32, x):
    """The kernels' evaluation of 2^x for fp32 x in a safe range: n by
    rounding with the 1.5 * 2^23 shift, f = x - n, Horner with FMAs, then n
    added to the exponent field."""
    x = np.asarray(x, dtype=np.float32)
    shift = np.float32(12582912.0)
    t = (x + shift).astype(np.float32)
    nf = (t - shift).astype(np.float32)
    f = (x - nf).astype(np.float32)
    p = np.full(f.shape, coef32[-1], dtype=np.float32)
    for c in coef32[-2::-1]:
        p = fp32_fma(p, f, c)
    bits = p.view(np.int32) + (nf.astype(np.int64).astype(np.int32) << 23)
    return bits.view(np.float32)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--degree", type=int, default=5)
    a = ap.parse_args()
    coef = remez_exp2(a.degree)
    coef32 = coef.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 400001)
    e_exact = np.abs(np.polyval(coef[::-1], f) / 2.0 ** f - 1).max()
    x = np.concatenate([np.linspace(-20, 8.5, 2_000_001, dtype=np.float32),
                        np.float32(np.random.default_rng(1).uniform(-120, 8.5, 1_000_000))])
    y = eval_fp32(coef32, x).astype(np.float64)
    e32 = np.abs(y / np.exp2(x.astype(np.float64)) - 1).max()
    print(f"degree {a.degree}: minimax relative error {e_exact:.3e} (2^{np.log2(e_exact):.2f}); "
          f"fp32 evaluation {e32:.3e} (2^{np.log2(e32):.2f})")
    for i, c in enumerate(coef32):
        print(f"  c{i} = {float(c)!r:>24}  ({float(c).hex()})")


if __name__ == "__main__":
    main()
