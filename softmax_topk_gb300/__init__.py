"""Python binding of libos_softmax.so (row-wise online softmax, fused softmax+TopK).

The C ABI (include/os_softmax.h) is wrapped with ctypes under the same names:
``os_softmax_fwd``, ``os_softmax_topk``, ``os_topk``, ``os_softmax_causal_fwd``,
``os_softmax_stats``, ``os_topk_sample``, ``os_attention_fwd``, ``os_softmax_fwd_path``,
``os_softmax_plan``, ``os_topk_plan``, ``os_exp_f32``, ``os_exp_pairs_f32``,
``os_exp_pairs_coarse_f32``, ``os_device_status``,
``os_set_wait_timeout_ns``, ``os_set_fault_injection``, ``os_status_string``.  They take raw
device pointers (ints) and a raw stream handle, exactly like the C functions,
and raise ``OsError`` on a non-OK status.

``softmax``, ``softmax_topk``, ``topk``, ``softmax_causal``, ``softmax_stats`` and
``attention`` are the
tensor-level conveniences: they take
torch CUDA tensors, allocate outputs with torch, pass the current torch
stream, and call the same C entry points.  PyTorch only provides memory and
streams; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is not built, importing this package
raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libos_softmax.so")

OS_F32, OS_BF16 = 0, 1
OS_PATH_AUTO, OS_PATH_WARP, OS_PATH_ONCHIP, OS_PATH_STREAM, OS_PATH_SAFE = 0, 1, 2, 3, 4
OS_PATH_STREAM_POLY = 5
PATHS = {"auto": OS_PATH_AUTO, "warp": OS_PATH_WARP, "onchip": OS_PATH_ONCHIP,
         "stream": OS_PATH_STREAM, "safe": OS_PATH_SAFE, "stream_poly": OS_PATH_STREAM_POLY}
STATUS = ["OS_OK", "OS_ERR_NULL", "OS_ERR_SHAPE", "OS_ERR_DTYPE", "OS_ERR_K", "OS_ERR_ALIAS",
          "OS_ERR_CUDA", "OS_ERR_TIMEOUT", "OS_ERR_PATH", "OS_ERR_ALIGN", "OS_ERR_VALUE"]
KMAX = 256


class OsError(RuntimeError):
    """A libos_softmax call returned a status other than OS_OK."""

    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS[status] if 0 <= status < len(STATUS) else str(status)
        super().__init__(f"{where}: {os_status_string(status)}")


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("vectors_per_thread", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("lanes_per_row", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("grid", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libos_softmax.so is not built ({LIB_PATH} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python softmax_topk_gb300/build.py` first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    lib.os_softmax_fwd.argtypes = [vp, vp, i64, i64, st, st, vp]
    lib.os_softmax_fwd_path.argtypes = [vp, vp, i64, i64, st, st, st, vp]
    lib.os_softmax_topk.argtypes = [vp, vp, vp, i64, i64, i32, vp]
    lib.os_topk.argtypes = [vp, vp, vp, i64, i64, i32, vp]
    lib.os_softmax_causal_fwd.argtypes = [vp, vp, i64, i64, i64, i64, st, st, vp]
    lib.os_softmax_stats.argtypes = [vp, vp, vp, vp, i64, i64, st, vp]
    lib.os_topk_sample.argtypes = [vp, vp, vp, vp, i64, i32, vp]
    lib.os_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, ctypes.c_float, i32, vp]
    lib.os_softmax_plan.argtypes = [i64, i64, st, st, st, ctypes.POINTER(Plan)]
    lib.os_topk_plan.argtypes = [i64, i64, i32, ctypes.POINTER(Plan)]
    lib.os_exp_f32.argtypes = [vp, vp, i64, vp]
    lib.os_exp_pairs_f32.argtypes = [vp, vp, i64, vp]
    lib.os_exp_pairs_coarse_f32.argtypes = [vp, vp, i64, vp]
    lib.os_device_status.argtypes = [vp]
    lib.os_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.os_set_fault_injection.argtypes = [i32]
    lib.os_status_string.argtypes = [st]
    lib.os_status_string.restype = ctypes.c_char_p
    for name in ("os_softmax_fwd", "os_softmax_fwd_path", "os_softmax_topk", "os_topk",
                 "os_softmax_causal_fwd", "os_softmax_stats", "os_topk_sample", "os_attention_fwd",
                 "os_softmax_plan",
                 "os_topk_plan", "os_exp_f32", "os_exp_pairs_f32", "os_exp_pairs_coarse_f32",
                 "os_device_status",
                 "os_set_wait_timeout_ns",
                 "os_set_fault_injection"):
        getattr(lib, name).restype = st
    return lib


_lib = _load()


def os_status_string(status: int) -> str:
    return _lib.os_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise OsError(status, where)


# ---------------------------------------------------------------- raw C entry points
def os_softmax_fwd(x: int, y: int, rows: int, cols: int, in_dtype: int, out_dtype: int,
                   stream: int | None) -> None:
    _check(_lib.os_softmax_fwd(x, y, rows, cols, in_dtype, out_dtype, stream), "os_softmax_fwd")


def os_softmax_fwd_path(x: int, y: int, rows: int, cols: int, in_dtype: int, out_dtype: int,
                        path: int, stream: int | None) -> None:
    _check(_lib.os_softmax_fwd_path(x, y, rows, cols, in_dtype, out_dtype, path, stream),
           "os_softmax_fwd_path")


def os_softmax_topk(x: int, vals: int, idx: int, rows: int, cols: int, K: int,
                    stream: int | None) -> None:
    _check(_lib.os_softmax_topk(x, vals, idx, rows, cols, K, stream), "os_softmax_topk")


def os_topk(x: int, vals: int, idx: int, rows: int, cols: int, K: int,
            stream: int | None) -> None:
    _check(_lib.os_topk(x, vals, idx, rows, cols, K, stream), "os_topk")


def os_softmax_causal_fwd(x: int, y: int, rows: int, cols: int, period: int, offset: int,
                          in_dtype: int, out_dtype: int, stream: int | None) -> None:
    _check(_lib.os_softmax_causal_fwd(x, y, rows, cols, period, offset, in_dtype, out_dtype,
                                      stream), "os_softmax_causal_fwd")


def os_softmax_stats(x: int, m: int | None, d: int | None, lse: int | None, rows: int, cols: int,
                     in_dtype: int, stream: int | None) -> None:
    _check(_lib.os_softmax_stats(x, m, d, lse, rows, cols, in_dtype, stream), "os_softmax_stats")


def os_topk_sample(vals: int, idx: int, u: int, out: int, rows: int, K: int,
                   stream: int | None) -> None:
    _check(_lib.os_topk_sample(vals, idx, u, out, rows, K, stream), "os_topk_sample")


def os_attention_fwd(q: int, k: int, v: int, o: int, lse: int | None, bh: int, n: int,
                     head_dim: int, scale: float, causal: int, stream: int | None) -> None:
    _check(_lib.os_attention_fwd(q, k, v, o, lse, bh, n, head_dim, scale, causal, stream),
           "os_attention_fwd")


def os_exp_f32(z: int, out: int, n: int, stream: int | None) -> None:
    _check(_lib.os_exp_f32(z, out, n, stream), "os_exp_f32")


def os_exp_pairs_f32(z: int, out: int, n: int, stream: int | None) -> None:
    _check(_lib.os_exp_pairs_f32(z, out, n, stream), "os_exp_pairs_f32")


def os_exp_pairs_coarse_f32(z: int, out: int, n: int, stream: int | None) -> None:
    _check(_lib.os_exp_pairs_coarse_f32(z, out, n, stream), "os_exp_pairs_coarse_f32")


def os_device_status(stream: int | None) -> None:
    """Synchronise `stream`; raise OsError(OS_ERR_TIMEOUT) if a device-side
    wait gave up since the last call."""
    _check(_lib.os_device_status(stream), "os_device_status")


def os_set_wait_timeout_ns(ns: int) -> None:
    _check(_lib.os_set_wait_timeout_ns(int(ns)), "os_set_wait_timeout_ns")


def os_set_fault_injection(mode: int) -> None:
    _check(_lib.os_set_fault_injection(int(mode)), "os_set_fault_injection")


def os_softmax_plan(rows: int, cols: int, in_dtype: int, out_dtype: int, path: int = 0) -> dict:
    p = Plan()
    _check(_lib.os_softmax_plan(rows, cols, in_dtype, out_dtype, path, ctypes.byref(p)),
           "os_softmax_plan")
    return p.as_dict()


def os_topk_plan(rows: int, cols: int, K: int) -> dict:
    p = Plan()
    _check(_lib.os_topk_plan(rows, cols, K, ctypes.byref(p)), "os_topk_plan")
    return p.as_dict()


# ---------------------------------------------------------------- torch conveniences
def _dtype_code(t) -> int:
    import torch
    if t == torch.float32:
        return OS_F32
    if t == torch.bfloat16:
        return OS_BF16
    raise TypeError(f"unsupported dtype {t}: float32 or bfloat16")


def _stream_handle(x) -> int:
    import torch
    return torch.cuda.current_stream(x.device).cuda_stream


class _OnDevice:
    """Make x's device current for the call (a no-op when it already is)."""

    def __init__(self, device):
        self.index = device.index

    def __enter__(self):
        import torch
        self.prev = torch.cuda.current_device()
        if self.prev != self.index:
            torch.cuda.set_device(self.index)

    def __exit__(self, *exc):
        import torch
        if self.prev != self.index:
            torch.cuda.set_device(self.prev)


def softmax(x, out_dtype=None, path: str | int = "auto", out=None):
    """Row-wise softmax of a 2-D CUDA tensor (fp32 or bf16) along its last dim."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    out_dtype = x.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    elif out.shape != x.shape or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be contiguous with x's shape and out_dtype")
    code = PATHS[path] if isinstance(path, str) else int(path)
    with _OnDevice(x.device):
        os_softmax_fwd_path(x.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1],
                            _dtype_code(x.dtype), _dtype_code(out_dtype), code,
                            _stream_handle(x))
    return out


def softmax_topk(x, K: int, vals=None, idx=None):
    """(probabilities fp32 [rows, K], column indices int32 [rows, K]) of each row's top K."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous() or x.dtype != torch.float32:
        raise ValueError("x must be a contiguous 2-D float32 CUDA tensor")
    rows = x.shape[0]
    if vals is None:
        vals = torch.empty((rows, K), dtype=torch.float32, device=x.device)
    if idx is None:
        idx = torch.empty((rows, K), dtype=torch.int32, device=x.device)
    with _OnDevice(x.device):
        os_softmax_topk(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, x.shape[1], K,
                        _stream_handle(x))
    return vals, idx


def topk(x, K: int, vals=None, idx=None):
    """(values fp32 [rows, K], column indices int32 [rows, K]) of each row's K largest
    values of x itself (no softmax)."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous() or x.dtype != torch.float32:
        raise ValueError("x must be a contiguous 2-D float32 CUDA tensor")
    rows = x.shape[0]
    if vals is None:
        vals = torch.empty((rows, K), dtype=torch.float32, device=x.device)
    if idx is None:
        idx = torch.empty((rows, K), dtype=torch.int32, device=x.device)
    with _OnDevice(x.device):
        os_topk(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, x.shape[1], K,
                _stream_handle(x))
    return vals, idx


def softmax_causal(x, period: int, offset: int = 0, out_dtype=None, out=None):
    """softmax(x) with columns c > (r mod period) + offset of row r masked in the kernel."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    out_dtype = x.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    with _OnDevice(x.device):
        os_softmax_causal_fwd(x.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1], int(period),
                              int(offset), _dtype_code(x.dtype), _dtype_code(out.dtype),
                              _stream_handle(x))
    return out


def softmax_stats(x, m=None, d=None, lse=None):
    """(m, d, lse) fp32 [rows] each: row maximum, sum of e^(x - m), and m + ln d
    (into the given tensors where passed)."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    rows = x.shape[0]
    outs = []
    for t in (m, d, lse):
        if t is None:
            t = torch.empty(rows, dtype=torch.float32, device=x.device)
        elif t.shape != (rows,) or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("m, d and lse must be contiguous float32 tensors of shape [rows]")
        outs.append(t)
    m, d, lse = outs
    with _OnDevice(x.device):
        os_softmax_stats(x.data_ptr(), m.data_ptr(), d.data_ptr(), lse.data_ptr(), rows,
                         x.shape[1], _dtype_code(x.dtype), _stream_handle(x))
    return m, d, lse


def topk_sample(vals, idx, u, out=None):
    """One column per row drawn from its K (probability, column) pairs; u: fp32 [rows] in [0, 1)."""
    import torch
    rows, K = vals.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.int32, device=vals.device)
    with _OnDevice(vals.device):
        os_topk_sample(vals.data_ptr(), idx.data_ptr(), u.data_ptr(), out.data_ptr(), rows, K,
                       _stream_handle(vals))
    return out


def softmax_topk_sample(x, K: int, u):
    """Fused softmax + TopK, then one draw per row: (samples, vals, idx)."""
    vals, idx = softmax_topk(x, K)
    return topk_sample(vals, idx, u), vals, idx


def attention(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
              want_lse: bool = True):
    """Attention forward on the tensor cores: (O, L) for bf16 CUDA tensors q, k, v
    of one shape [..., n, head_dim] (leading dims are the batch x head slices),
    head_dim 64 or 128.  O has q's shape (bf16); L is fp32 [..., n], or None
    when ``want_lse`` is false.  ``scale`` defaults to 1/sqrt(head_dim)."""
    import torch
    for t_ in (q, k, v):
        if not t_.is_cuda or t_.dtype != torch.bfloat16 or not t_.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() < 2:
        raise ValueError("q, k, v must share one shape [..., n, head_dim]")
    n, hd = q.shape[-2], q.shape[-1]
    bh = q.numel() // max(n * hd, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    s = (1.0 / hd ** 0.5) if scale is None else float(scale)
    with _OnDevice(q.device):
        os_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, bh, n, hd, s, int(causal),
                         _stream_handle(q))
    return out, lse


def exp(z, pairs: bool = False, coarse: bool = False):
    """e^z elementwise (fp32 CUDA tensor) with the library's own exponential:
    the accurate scalar routine, or (pairs=True, z <= 0) the per-element
    exponential of the streaming kernel's fp32 results, or (pairs=True,
    coarse=True) that of its bf16 results before their rounding."""
    import torch
    if not z.is_cuda or z.dtype != torch.float32 or not z.is_contiguous():
        raise ValueError("z must be a contiguous float32 CUDA tensor")
    out = torch.empty_like(z)
    fn = (os_exp_pairs_coarse_f32 if coarse else os_exp_pairs_f32) if pairs else os_exp_f32
    with _OnDevice(z.device):
        fn(z.data_ptr(), out.data_ptr(), z.numel(), _stream_handle(z))
    return out


def plan(x_shape, in_dtype=OS_F32, out_dtype=None, path: str | int = "auto") -> dict:
    out_dtype = in_dtype if out_dtype is None else out_dtype
    code = PATHS[path] if isinstance(path, str) else int(path)
    return os_softmax_plan(int(x_shape[0]), int(x_shape[1]), in_dtype, out_dtype, code)
