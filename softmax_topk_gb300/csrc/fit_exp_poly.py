"""Derivation of the polynomials of the library's fp32 exponentials in
kernels/ops.cuh: e^r for exp1 (os_exp_f32, merge rescale factors, TopK
values), and 2^f for the per-element exponentials of the streaming softmax
kernels (exp_biased_pair, second part of this file: degree 5 for fp32
results, degree 3 for bf16 results).

The kernels evaluate e^z as 2^n * p(r) with n = rint(z * log2 e) and
r = z - n ln2 (Cody & Waite, "Software Manual for the Elementary Functions",
1980: argument reduction with ln2 split into an exactly representable high
part and a small low part).  After the reduction |r| <= ln2/2 plus the slack
caused by rounding log2 e to fp32, so p is fitted on [-A, A] with
A = 0.3466 + 2e-4.

p(r) = 1 + c1 r + ... + c6 r^6 minimises max |p(r) e^-r - 1| (relative
error, with p(0) = 1 exactly so that e^0 is exactly 1).  The fit is a
Lawson iteratively-reweighted least-squares solve on 4001 Chebyshev points,
which converges to the minimax (equioscillating) solution; the coefficients
are then rounded to fp32.  Running this file prints them and the fit's
relative error (about 2e-9, i.e. 0.03 ulp; the fp32 evaluation adds roughly
one ulp of rounding, which the library's GPU tests measure against float64).

This script is documentation of where the constants in kernels/ops.cuh come
from; nothing imports it.
"""
import numpy as np

A = 0.3466 + 2e-4
DEGREE = 6


def lawson_fit(degree: int, iters: int = 60, fn=np.exp, half_width: float = A):
    r = np.cos(np.linspace(0.0, np.pi, 4001)) * half_width
    f = fn(r)
    basis = np.stack([r ** k for k in range(1, degree + 1)], axis=1) / f[:, None]
    target = (f - 1.0) / f
    w = np.ones_like(r)
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(basis * sw[:, None], target * sw, rcond=None)
        err = np.abs(basis @ c - target)
        w = w * err
        w /= w.sum()
    return np.concatenate([[1.0], c]), float(err.max())


# 2^f on [-1/2, 1/2] (the per-element exponential of fp32 results):
# e^z = 2^n 2^f with n = rint(z log2 e) and f = z log2 e - n, so the fit is of
# 2^f itself, again relative and with p(0) = 1 exactly; degree 5 gives about
# 9e-8 (1.1e-7 once the coefficients are rounded to fp32).
DEGREE_2F = 5
# Where results are rounded to bf16 (relative rounding 2^-9), degree 3 on the
# same interval is enough: about 1.0e-4 with fp32 coefficients.
DEGREE_2F_BF16 = 3


if __name__ == "__main__":
    coeffs, err = lawson_fit(DEGREE)
    print(f"e^r, degree {DEGREE}: max relative error {err:.3e}")
    for k, c in enumerate(coeffs):
        c32 = np.float32(c)
        print(f"c{k} = {c32!r}  (0x{int(c32.view(np.uint32)):08x})")
    for deg in (DEGREE_2F, DEGREE_2F_BF16):
        coeffs, err = lawson_fit(deg, iters=80, fn=np.exp2, half_width=0.5)
        print(f"2^f, degree {deg}: max relative error {err:.3e}")
        for k, c in enumerate(coeffs):
            c32 = np.float32(c)
            print(f"e{deg}_{k} = {c32!r}  (0x{int(c32.view(np.uint32)):08x})")
