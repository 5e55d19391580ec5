"""The forward kernels' FMA-pipe exponential (exp2_poly in fa_fwd_common.cuh): its
coefficients match the generator, and the float32 algorithm (round-to-
nearest split by the 1.5*2^23 trick, degree-4 polynomial on [-1/2, 1/2],
exponent-field add) stays within its stated error bound against 2^x."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_25_gb300", "csrc")


def kernel_coefficients():
    text = open(os.path.join(CSRC, "fa_fwd_common.cuh")).read()
    vals = dict(re.findall(r"\bkExp2C([0-4]) = ([-+0-9.e]+)f", text))
    return np.array([float(vals[str(i)]) for i in range(5)], np.float32)


def emulate(x, c):
    """float32 replay of exp2_poly, operation by operation."""
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(f32)
    n = (t - f32(12582912.0)).astype(f32)
    r = (x - n).astype(f32)
    q = c[4]
    for k in (3, 2, 1, 0):
        q = (q * r + c[k]).astype(f32)  # fmaf rounds once; this rounds twice (looser)
    ni = t.view(np.int32) - np.int32(0x4B400000)
    return (q.view(np.int32) + (ni << 23)).view(f32)


def test_coefficients_match_generator():
    sys.path.insert(0, CSRC)
    import gen_exp2_poly
    want = gen_exp2_poly.coefficients().astype(np.float32)
    np.testing.assert_array_equal(kernel_coefficients(), want)


def test_polynomial_error_bound_on_reduced_interval():
    c = kernel_coefficients().astype(np.float64)
    f = np.linspace(-0.5, 0.5, 200001)
    p = np.polyval(c[::-1], f)
    rel = np.abs(p / np.exp2(f) - 1.0)
    assert rel.max() < 4e-6


def test_float32_algorithm_matches_exp2():
    c = kernel_coefficients()
    x = np.concatenate([np.linspace(-126.0, 9.0, 400001), -np.arange(0, 126, 1.0),
                        np.arange(0.5, 9, 1.0)]).astype(np.float32)
    got = emulate(x, c).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1e-5, rel.max()
    # below the clamp the result is tiny and positive, never garbage
    tiny = emulate(np.array([-200.0, -1e30, -np.inf], np.float32), c)
    assert np.all(tiny >= 0) and np.all(tiny < 1e-37)
