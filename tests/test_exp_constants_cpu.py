"""The exponential's polynomial constants in kernels/ops.cuh are the fp32
roundings of the fits that csrc/fit_exp_poly.py derives (e^r, degree 6, for
the accurate scalar routine; 2^f, degree 5 and 3, for the streaming kernel's
per-element exponential of fp32 and bf16 results), bit for bit."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "softmax_topk_gb300", "csrc")


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp_poly",
                                                  os.path.join(CSRC, "fit_exp_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _constants():
    text = open(os.path.join(CSRC, "kernels", "ops.cuh")).read()
    return {name: np.float32(float(val)) for name, val in
            re.findall(r"\b(c[1-6]|e5_[1-5]|e3_[1-3])\s*=\s*([-+0-9.eE]+)f", text)}


def test_exp_polynomial_constants_match_their_fits():
    fit = _fit_module()
    consts = _constants()
    c, err = fit.lawson_fit(fit.DEGREE)
    assert err < 3e-9
    for k in range(1, fit.DEGREE + 1):
        assert np.float32(c[k]) == consts[f"c{k}"], (k, np.float32(c[k]), consts[f"c{k}"])
    e, err2 = fit.lawson_fit(fit.DEGREE_2F, iters=80, fn=np.exp2, half_width=0.5)
    assert err2 < 1e-7
    for k in range(1, fit.DEGREE_2F + 1):
        assert np.float32(e[k]) == consts[f"e5_{k}"], (k, np.float32(e[k]), consts[f"e5_{k}"])
    e3, err3 = fit.lawson_fit(fit.DEGREE_2F_BF16, iters=80, fn=np.exp2, half_width=0.5)
    assert err3 < 1.02e-4
    for k in range(1, fit.DEGREE_2F_BF16 + 1):
        assert np.float32(e3[k]) == consts[f"e3_{k}"], (k, np.float32(e3[k]), consts[f"e3_{k}"])


def test_exp2_fit_error_with_fp32_coefficients():
    """Evaluated in float64 with the fp32 constants, 2^f is within 1.1e-7 on
    [-1/2, 1/2] (the figure the kernels' error statements use)."""
    consts = _constants()
    f = np.linspace(-0.5, 0.5, 200001)
    p = np.full_like(f, float(consts["e5_5"]))
    for k in (4, 3, 2, 1):
        p = p * f + float(consts[f"e5_{k}"])
    p = p * f + 1.0
    assert np.abs(p / np.exp2(f) - 1).max() <= 1.1e-7


def test_exp2_degree3_fit_error_with_fp32_coefficients():
    """The bf16 results' fit, evaluated in float64 with its fp32 constants, is
    within 1.02e-4 of 2^f on [-1/2, 1/2]: with bf16's 2^-9 rounding the
    result stays far inside the 8e-3 tolerance."""
    consts = _constants()
    f = np.linspace(-0.5, 0.5, 200001)
    p = np.full_like(f, float(consts["e3_3"]))
    for k in (2, 1):
        p = p * f + float(consts[f"e3_{k}"])
    p = p * f + 1.0
    assert np.abs(p / np.exp2(f) - 1).max() <= 1.02e-4


def test_biased_exponent_arithmetic():
    """The integer step of the FMA-pipe exponential, restated on the host in
    fp32: u = fl(z log2e + 1.5 * 2^23 + 66) holds n + 66 in its low bits, and
    adding u's bits shifted by 23 to p's bits multiplies p by 2^(n + 66); the
    clamp at z = -110 keeps the exponent field of the result >= 2."""
    text = open(os.path.join(CSRC, "kernels", "ops.cuh")).read()
    biased = np.float32(float(re.search(r"kBiasedRound = ([0-9.]+)f", text).group(1)))
    clamp = np.float32(float(re.search(r"kZClamp = (-[0-9.]+)f", text).group(1)))
    log2e = np.float32(float(re.search(r"kLog2e = ([0-9.e+-]+)f", text).group(1)))
    assert biased == np.float32(1.5 * 2 ** 23 + 66)
    z = np.concatenate([np.linspace(float(clamp), 0.0, 100001, dtype=np.float32),
                        np.array([clamp, -0.0, 0.0], dtype=np.float32)])
    # the FMA: exact product and sum (within float64's 53 bits here), one rounding
    u = np.float32(np.float64(z) * np.float64(log2e) + np.float64(biased))
    n = np.rint(np.float64(z) * np.float64(log2e))
    assert np.array_equal(np.float64(u) - 1.5 * 2 ** 23 - 66, n)
    for p in (np.float32(0.70710677), np.float32(1.0), np.float32(1.4142135)):
        bits = (p.view(np.uint32).astype(np.uint64) +
                (u.view(np.uint32).astype(np.uint64) << np.uint64(23))) % 2 ** 32
        q = bits.astype(np.uint32).view(np.float32).astype(np.float64)
        assert np.array_equal(q, np.float64(p) * np.exp2(n + 66))
        assert ((bits >> np.uint64(23)) & np.uint64(255)).min() >= 2
