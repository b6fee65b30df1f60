"""The 2^x polynomial emulation and its accuracy table.

Test infrastructure only (see the package docstring).

Source: "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", abstract and Table 2; "FlashAttention 3 and 4:
When the Bottleneck Moves", section 3.2 (first change); "Attention at Scale",
FlashAttention-4 paragraph ("software-emulated exp2 ... integer bit
manipulation").

Method: 2^x = 2^floor(x) * 2^f with f = x - floor(x) in [0, 1).  2^f is a
polynomial of low degree; 2^floor(x) is applied by adding floor(x) to the
binary exponent.  The pages print the polynomial's error on [0, 1) (Table 2)
but not its coefficients.

Reading: the polynomial is the degree-n minimax fit of 2^f on [0, 1] in
relative error with the constant term fixed to 1 (so integer x is exact).
This reading reproduces Table 2's mean errors to within a few per cent for
degrees 3 and 4; the CPU tests pin it there.  The fit below is our own Remez
exchange in FP64.
"""
from __future__ import annotations

import numpy as np


def fit_exp2_poly(degree: int, iters: int = 60, grid_points: int = 200_001) -> np.ndarray:
    """Minimax (relative error) polynomial for 2^f on [0, 1] with p(0) = 1.

    p(f) = 1 + c1 f + ... + cn f^n.  Remez exchange on the n free coefficients
    and the levelled error E: at n + 1 reference points x_i solve
    p(x_i) - 2^x_i = (-1)^i E 2^x_i, then move the references to the extrema
    of the relative error on a dense grid.  Returns [1, c1, ..., cn] (FP64,
    lowest degree first).
    """
    n = degree
    grid = np.linspace(0.0, 1.0, grid_points)
    x = 0.5 - 0.5 * np.cos(np.pi * (np.arange(n + 1) + 0.5) / (n + 1))
    coeffs = None
    for _ in range(iters):
        f = np.exp2(x)
        a = np.empty((n + 1, n + 1))
        for j in range(1, n + 1):
            a[:, j - 1] = x ** j
        a[:, n] = ((-1.0) ** np.arange(n + 1)) * f
        sol = np.linalg.solve(a, f - 1.0)
        coeffs = np.concatenate([[1.0], sol[:n]])
        err = relative_error_f64(coeffs, grid)
        sgn = np.where(err >= 0, 1, -1)
        segs = np.split(np.arange(grid_points), np.nonzero(np.diff(sgn))[0] + 1)
        ext = np.array([grid[sg[np.argmax(np.abs(err[sg]))]] for sg in segs])
        if len(ext) > n + 1:
            keep = np.sort(np.argsort(-np.abs(relative_error_f64(coeffs, ext)))[: n + 1])
            ext = ext[keep]
        if len(ext) < n + 1:
            break
        if np.max(np.abs(ext - x)) < 1e-12:
            break
        x = ext
    return coeffs


def relative_error_f64(coeffs: np.ndarray, f: np.ndarray) -> np.ndarray:
    """(p(f) - 2^f) / 2^f in FP64."""
    return (np.polyval(coeffs[::-1], f) - np.exp2(f)) / np.exp2(f)


def eval_poly_f32(coeffs: np.ndarray, f: np.ndarray) -> np.ndarray:
    """Horner evaluation with FP32 coefficients and FP32 fused multiply-adds.

    Each step computes p * f + c exactly in FP64 (the product of two FP32
    numbers is exact there) and rounds once to FP32, as a fused multiply-add does.
    """
    c32 = np.asarray(coeffs, dtype=np.float32)
    f32 = np.asarray(f, dtype=np.float32).astype(np.float64)
    p = np.full(f32.shape, c32[-1], dtype=np.float32)
    for c in c32[-2::-1]:
        p = (p.astype(np.float64) * f32 + np.float64(c)).astype(np.float32)
    return p


def exp2_emulated(coeffs: np.ndarray, x: np.ndarray) -> np.ndarray:
    """2^x for FP32 x by the method: 2^floor(x) times the polynomial at the fraction."""
    x32 = np.asarray(x, dtype=np.float32)
    n = np.floor(x32)
    frac = (x32 - n).astype(np.float32)
    return np.ldexp(eval_poly_f32(coeffs, frac), n.astype(np.int32))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to bfloat16 (nearest, ties to even), returned as FP64."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)) << np.uint32(16)
    return r.view(np.float32).astype(np.float64)


def accuracy_row(values_f32: np.ndarray, f: np.ndarray) -> dict:
    """Max and mean relative error of FP32 results and of their bfloat16 rounding vs FP64 2^f."""
    exact = np.exp2(np.asarray(f, dtype=np.float32).astype(np.float64))
    r32 = np.abs(values_f32.astype(np.float64) - exact) / exact
    rbf = np.abs(round_bf16(values_f32) - exact) / exact
    return {"fp32_max": float(r32.max()), "fp32_mean": float(r32.mean()),
            "bf16_max": float(rbf.max()), "bf16_mean": float(rbf.mean())}


def accuracy_table(degrees=(3, 4, 5), n: int = 4_000_000, seed: int = 0) -> dict:
    """Table 2's experiment: ``n`` uniform inputs on [0, 1) (FP32), each degree's fit.

    The inputs are FP32 rounds of uniform FP64 draws; values that round to 1.0
    are dropped so the domain stays [0, 1).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    f = rng.random(n).astype(np.float32)
    f = f[f < 1.0]
    table = {"ideal": accuracy_row(f_ideal := np.exp2(f.astype(np.float64)).astype(np.float32), f)}
    del f_ideal
    for d in degrees:
        table[f"degree{d}"] = accuracy_row(eval_poly_f32(fit_exp2_poly(d), f), f)
    return table
