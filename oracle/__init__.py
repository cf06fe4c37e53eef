"""float64 CPU oracle for row-wise softmax and fused softmax+TopK.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C99, IEEE double, host libm
``exp``); this module compiles it with gcc on first use and wraps it with
ctypes/numpy.  Inputs of any real dtype are widened to float64 exactly
(bf16 and fp32 values are exact in double) before the C code sees them.

Functions and the passages they follow are listed in ``oracle.c``'s header:
``softmax`` (three-pass safe softmax), ``row_stats`` ((m, d) by definition),
``online_stats`` (the single-pass recurrence), ``combine`` (the binary
operator on (m, d) with identity (-inf, 0)), ``topk`` (full sort by
logit descending, index ascending; v = e^(u - m)/d), ``lse`` (m + ln d),
``causal_mask`` / ``softmax_causal`` (the causal mask, then softmax),
``topk_sample`` (one draw per row from its top-K pairs) and ``attention``
(softmax(scale Q K^T) V and the logsumexp of each query row).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dbl_p = ctypes.POINTER(ctypes.c_double)
_i32_p = ctypes.POINTER(ctypes.c_int32)
_i64_p = ctypes.POINTER(ctypes.c_int64)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, defines: tuple = ()) -> str:
    """Compile ``src`` into a shared library at ``out`` with gcc (OpenMP on)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp",
           *[f"-D{d}" for d in defines], src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle()
    return _LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (or another build of the same source at ``path``)."""
    lib = ctypes.CDLL(path or build())
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_row_stats_f64.argtypes = [_dbl_p, _dbl_p, _dbl_p, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_softmax_f64.argtypes = [_dbl_p, _dbl_p, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_online_stats_f64.argtypes = [_dbl_p, ctypes.c_int64, _dbl_p, _dbl_p]
    lib.oracle_combine_f64.argtypes = [ctypes.c_double] * 4 + [_dbl_p, _dbl_p]
    lib.oracle_topk_f64.argtypes = [_dbl_p, _dbl_p, _i32_p, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int32]
    lib.oracle_topk_f64.restype = ctypes.c_int
    lib.oracle_lse_f64.argtypes = [_dbl_p, _dbl_p, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_causal_mask_f64.argtypes = [_dbl_p, _dbl_p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64]
    lib.oracle_topk_sample_f64.argtypes = [_dbl_p, _i32_p, _dbl_p, _i32_p, ctypes.c_int64,
                                           ctypes.c_int32]
    lib.oracle_attention_f64.argtypes = [_dbl_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_double,
                                                                              ctypes.c_int]
    lib.oracle_attention_rows_f64.argtypes = [_dbl_p] * 3 + [_i64_p, _i64_p] + \
        [ctypes.c_int64] * 3 + [ctypes.c_double, ctypes.c_int, _dbl_p, _dbl_p]
    return lib


def _get() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load()
    return _lib


def _as_rows(x) -> np.ndarray:
    """Widen to a C-contiguous float64 matrix (exact for fp32 and bf16 data)."""
    if hasattr(x, "detach"):  # a torch tensor: widen on its device-independent CPU copy
        x = x.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if a.ndim == 1:
        a = a[None, :]
    if a.ndim != 2:
        raise ValueError("oracle inputs are rows: a 1-D or 2-D array")
    return a


def _p(a: np.ndarray, t=_dbl_p):
    return a.ctypes.data_as(t)


def num_threads(lib: ctypes.CDLL | None = None) -> int:
    return (lib or _get()).oracle_num_threads()


def set_num_threads(n: int, lib: ctypes.CDLL | None = None) -> None:
    """Threads of the oracle's row loops from now on (timing only: the
    arithmetic of a row does not depend on it)."""
    (lib or _get()).oracle_set_num_threads(int(n))


def softmax(x, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """float64 softmax of each row of ``x`` (three-pass safe softmax)."""
    a = _as_rows(x)
    y = np.empty_like(a)
    (lib or _get()).oracle_softmax_f64(_p(a), _p(y), a.shape[0], a.shape[1])
    return y


def row_stats(x, lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Per-row (m, d): the row maximum and sum_j e^(x_j - m)."""
    a = _as_rows(x)
    m = np.empty(a.shape[0])
    d = np.empty(a.shape[0])
    (lib or _get()).oracle_row_stats_f64(_p(a), _p(m), _p(d), a.shape[0], a.shape[1])
    return m, d


def online_stats(x, lib: ctypes.CDLL | None = None) -> tuple[float, float]:
    """(m, d) of a 1-D sequence by the element-by-element recurrence."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
    m = ctypes.c_double()
    d = ctypes.c_double()
    (lib or _get()).oracle_online_stats_f64(_p(a), a.size, ctypes.byref(m), ctypes.byref(d))
    return m.value, d.value


def combine(s1, s2, lib: ctypes.CDLL | None = None) -> tuple[float, float]:
    """(m1, d1) (+) (m2, d2)."""
    m = ctypes.c_double()
    d = ctypes.c_double()
    (lib or _get()).oracle_combine_f64(float(s1[0]), float(s1[1]), float(s2[0]), float(s2[1]),
                                       ctypes.byref(m), ctypes.byref(d))
    return m.value, d.value


def topk(x, K: int, lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Top-K (probability float64, index int32) of each row, best first."""
    a = _as_rows(x)
    rows, cols = a.shape
    vals = np.empty((rows, K))
    idx = np.empty((rows, K), dtype=np.int32)
    rc = (lib or _get()).oracle_topk_f64(_p(a), _p(vals), _p(idx, _i32_p), rows, cols, K)
    if rc != 0:
        raise ValueError(f"oracle topk rejected K={K} for {cols} columns")
    return vals, idx


def lse(x, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Per-row log-sum-exp, m + ln d (-inf for rows that are all -inf)."""
    a = _as_rows(x)
    out = np.empty(a.shape[0])
    (lib or _get()).oracle_lse_f64(_p(a), _p(out), a.shape[0], a.shape[1])
    return out


def causal_mask(x, period: int, offset: int = 0, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """x with the entries c > (r mod period) + offset of row r set to -inf."""
    a = _as_rows(x)
    out = np.empty_like(a)
    (lib or _get()).oracle_causal_mask_f64(_p(a), _p(out), a.shape[0], a.shape[1], int(period),
                                           int(offset))
    return out


def softmax_causal(x, period: int, offset: int = 0, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """float64 softmax of each row of ``x`` under the causal mask above."""
    return softmax(causal_mask(x, period, offset, lib=lib), lib=lib)


def topk_sample(vals, idx, u, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """One column per row from its K (value, index) pairs: the smallest k whose
    partial sum exceeds u times the total (sums in index order)."""
    v = _as_rows(vals)
    ix = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(v.shape))
    uu = np.ascontiguousarray(np.asarray(u, dtype=np.float64).ravel())
    if uu.size != v.shape[0]:
        raise ValueError("one u per row")
    out = np.empty(v.shape[0], dtype=np.int32)
    (lib or _get()).oracle_topk_sample_f64(_p(v), _p(ix, _i32_p), _p(uu), _p(out, _i32_p),
                                           v.shape[0], v.shape[1])
    return out


def _as_heads(x) -> np.ndarray:
    """Widen a [bh, n, dh] array (or tensor) to C-contiguous float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if a.ndim == 2:
        a = a[None]
    if a.ndim != 3:
        raise ValueError("attention inputs are [bh, n, dh] (or [n, dh])")
    return a


def attention(q, k, v, scale: float | None = None, causal: bool = False,
              lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, np.ndarray]:
    """float64 softmax(scale Q K^T) V per (batch, head) slice and the logsumexp
    L = m + ln d of each query row; with ``causal`` query i sees keys j <= i.
    ``scale`` defaults to 1/sqrt(dh).  Returns (O [bh, n, dh], L [bh, n])."""
    a, b, c = _as_heads(q), _as_heads(k), _as_heads(v)
    if a.shape != b.shape or a.shape != c.shape:
        raise ValueError("q, k and v must have one shape [bh, n, dh]")
    bh, n, dh = a.shape
    s = 1.0 / np.sqrt(dh) if scale is None else float(scale)
    o = np.empty_like(a)
    lse_out = np.empty((bh, n))
    (lib or _get()).oracle_attention_f64(_p(a), _p(b), _p(c), _p(o), _p(lse_out), bh, n, dh, s,
                                         int(bool(causal)))
    return o, lse_out


def attention_rows(q_rows, k, v, slices, rows, scale: float | None = None, causal: bool = False,
                   lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, np.ndarray]:
    """The attention oracle for selected query rows only: ``q_rows`` [p, dh] holds
    query ``rows[p]`` of slice ``slices[p]``; k, v are the full [bh, n, dh].
    Returns (O [p, dh], L [p])."""
    b, c = _as_heads(k), _as_heads(v)
    if b.shape != c.shape:
        raise ValueError("k and v must have one shape [bh, n, dh]")
    bh, n, dh = b.shape
    a = _as_heads(q_rows).reshape(-1, dh)
    sl = np.ascontiguousarray(np.asarray(slices, dtype=np.int64).ravel())
    rw = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    if not (len(sl) == len(rw) == a.shape[0]):
        raise ValueError("one (slice, row) pair per query row")
    if len(sl) and (sl.min() < 0 or sl.max() >= bh or rw.min() < 0 or rw.max() >= n):
        raise ValueError("(slice, row) pair out of range")
    s = 1.0 / np.sqrt(dh) if scale is None else float(scale)
    o = np.empty((len(sl), dh))
    lse_out = np.empty(len(sl))
    (lib or _get()).oracle_attention_rows_f64(_p(a), _p(b), _p(c), _p(sl, _i64_p), _p(rw, _i64_p),
                                              len(sl), n, dh, s, int(bool(causal)), _p(o),
                                              _p(lse_out))
    return o, lse_out
