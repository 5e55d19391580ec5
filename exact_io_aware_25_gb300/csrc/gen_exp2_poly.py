"""Coefficients of the polynomial 2^f ~ p(f) on f in [-1/2, 1/2] used by the
forward kernel to compute part of its exponentials on the FMA pipe.

Method: interpolation of 2^f at the 5 Chebyshev nodes of [-1/2, 1/2]
(a near-minimax polynomial; the interpolation error is bounded by
max|d^5/df^5 2^f| / (5! * 2^4) * (1/2)^5 = 2^(1/2) (ln 2)^5 / 61440 ~ 3.7e-6).
The printed coefficients (c0 + c1 f + ... + c4 f^4, rounded to float32) are
copied into fa_fwd.cu; tests/test_exp2_poly.py re-evaluates them.
"""
import numpy as np

DEGREE = 4


def coefficients(degree: int = DEGREE) -> np.ndarray:
    k = np.arange(degree + 1)
    nodes = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * (degree + 1)))
    V = np.vander(nodes, degree + 1, increasing=True)
    return np.linalg.solve(V, np.exp2(nodes))


if __name__ == "__main__":
    c = coefficients().astype(np.float32)
    for i, x in enumerate(c):
        print(f"c{i} = {float(x):.9e}f")
