"""Element-by-element comparison of library outputs with the float64 oracle.

Rules (fp32 outputs; the same with the bf16 tolerance for bf16 outputs):
  * where the oracle's probability is >= FLT_MIN (2^-126), the relative error
    |y - y_ref| / y_ref must be <= tol (1e-5 fp32, 8e-3 bf16);
  * where it is below FLT_MIN (deep underflow, e.g. e^-137 / d), the output
    must be in [0, FLT_MIN];
  * where the input is -inf the output must be exactly +0;
  * every row's outputs sum to 1 within sum_tol.
"""
import numpy as np

FLT_MIN = float(np.finfo(np.float32).tiny)
TOL = {"f32": 1e-5, "bf16": 8e-3}
# a row of n bf16 outputs carries at most 2^-9 relative rounding per term
SUM_TOL = {"f32": 1e-5, "bf16": 1e-2}


def softmax_errors(x64: np.ndarray, y: np.ndarray, ref: np.ndarray) -> dict:
    y = y.astype(np.float64)
    big = ref >= FLT_MIN
    rel = np.zeros_like(ref)
    rel[big] = np.abs(y[big] - ref[big]) / ref[big]
    tiny_bad = (~big) & ((y < 0) | (y > FLT_MIN))
    neg_inf = np.isneginf(x64)
    inf_bad = neg_inf & ~((y == 0) & ~np.signbit(y))
    sums = y.sum(axis=1)
    return {"max_rel": float(rel.max()) if rel.size else 0.0,
            "argmax_rel": np.unravel_index(int(np.argmax(rel)), rel.shape) if rel.size else None,
            "tiny_bad": int(tiny_bad.sum()), "neg_inf_bad": int(inf_bad.sum()),
            "max_sum_err": float(np.abs(sums - 1.0).max()) if sums.size else 0.0,
            "nan": int(np.isnan(y).sum())}


def assert_softmax_close(x64, y, ref, out_dtype: str, label: str = "") -> dict:
    e = softmax_errors(x64, y, ref)
    tol, stol = TOL[out_dtype], SUM_TOL[out_dtype]
    msg = f"{label}: {e}"
    assert e["nan"] == 0, msg
    assert e["max_rel"] <= tol, msg
    assert e["tiny_bad"] == 0, msg
    assert e["neg_inf_bad"] == 0, msg
    assert e["max_sum_err"] <= stol, msg
    return e


def assert_topk_equal(vals, idx, ref_vals, ref_idx, label: str = "") -> None:
    idx = np.asarray(idx)
    ref_idx = np.asarray(ref_idx)
    bad = np.argwhere(idx != ref_idx)
    assert bad.size == 0, f"{label}: {len(bad)} index mismatches, first at {bad[:3].tolist()}: " \
                          f"got {idx[tuple(bad[0])]} want {ref_idx[tuple(bad[0])]}"
    vals = np.asarray(vals, dtype=np.float64)
    big = ref_vals >= FLT_MIN
    rel = np.abs(vals[big] - ref_vals[big]) / ref_vals[big]
    assert rel.size == 0 or rel.max() <= TOL["f32"], f"{label}: max rel {rel.max():.3e}"
    small = ~big
    assert np.all((vals[small] >= 0) & (vals[small] <= FLT_MIN)), f"{label}: tiny values"
