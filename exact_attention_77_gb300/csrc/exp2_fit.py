"""Coefficients of the 2^f polynomials used by the kernels (f in [0, 1)).

The kernels evaluate 2^x as 2^floor(x) * p(x - floor(x)), the split described
in "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling" (abstract; Table 2 gives the error of degrees 3 to 5).  The
pages print no coefficients, so they are fitted here: p(0) = 1 is fixed
(integer arguments come out exact) and the relative error max |p/2^f - 1| on
[0, 1] is minimised by Lawson's iteratively reweighted least squares, which
converges to the minimax solution.

Run ``python exp2_fit.py`` to print the constants pasted into sm103.cuh (the
cubic the forward kernel uses) and probes.cu (degrees 4 and 5).
"""
import numpy as np


def lawson_fit(degree: int, iters: int = 4000, points: int = 4001) -> np.ndarray:
    x = 0.5 - 0.5 * np.cos(np.linspace(0.0, np.pi, points))  # Chebyshev-spaced nodes on [0, 1]
    target = np.exp2(x)
    basis = np.stack([x ** j for j in range(1, degree + 1)], axis=1) / target[:, None]
    rhs = (target - 1.0) / target  # relative residual of p = 1 + sum c_j x^j
    w = np.full(points, 1.0 / points)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(basis * sw[:, None], rhs * sw, rcond=None)
        err = np.abs(basis @ c - rhs)
        w = w * err
        w /= w.sum()
    return np.concatenate([[1.0], c])


if __name__ == "__main__":
    for d in (3, 4, 5):
        c = lawson_fit(d)
        g = np.linspace(0, 1, 100001)
        rel = np.abs(np.polyval(c[::-1], g) / np.exp2(g) - 1).max()
        print(f"degree {d}: max rel {rel:.4e}  coeffs", ", ".join(f"{v:.9g}f" for v in c[1:]))
