"""The exponential's polynomial constants in kernels/ops.cuh are the fp32
roundings of the fits that csrc/fit_exp_poly.py derives (e^r, degree 6, for
the accurate scalar routine; 2^f, degree 5, for the streaming kernel's
per-element exponential), bit for bit."""
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
            re.findall(r"\b(c[1-6]|e5_[1-5])\s*=\s*([-+0-9.eE]+)f", text)}


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
