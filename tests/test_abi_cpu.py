"""The C ABI on a machine without a GPU: the library loads, exports every
function include/*.h declares, and rejects bad arguments before touching the
device.  No kernel is launched here."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "softmax_topk_gb300", "lib", "libos_softmax.so")

F32, BF16 = 0, 1
OK, NULL, SHAPE, DTYPE, KERR, ALIAS, CUDA, TIMEOUT, PATH, ALIGN, VALUE = range(11)


def _ensure_built():
    import __graft_entry__
    __graft_entry__._builder().build()


@pytest.fixture(scope="module")
def lib():
    _ensure_built()
    import softmax_topk_gb300 as st
    return st._lib


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(os_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("os_softmax_fwd", "os_softmax_topk", "os_attention_fwd", "os_status_string"):
        assert required in names, names


def test_every_declared_function_is_exported(lib):
    raw = ctypes.CDLL(LIB)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    import softmax_topk_gb300 as st
    for code, name in enumerate(st.STATUS):
        assert st.os_status_string(code).startswith(name)
    assert st.os_status_string(99) == "unknown os_status"


A, B, C = 0x10000, 0x4000000, 0x8000000  # disjoint fake device addresses, 16-byte aligned


def test_softmax_argument_errors(lib):
    f = lib.os_softmax_fwd_path
    assert f(A, B, 4, 8, 2, F32, 0, None) == DTYPE
    assert f(A, B, 4, 8, F32, -1, 0, None) == DTYPE
    assert f(A, B, -1, 8, F32, F32, 0, None) == SHAPE
    assert f(A, B, 4, 0, F32, F32, 0, None) == SHAPE
    assert f(A, B, 4, 2 ** 31, F32, F32, 0, None) == SHAPE
    assert f(A, B, 2 ** 62, 2 ** 20, F32, F32, 0, None) == SHAPE
    assert f(A, B, 4, 8, F32, F32, 7, None) == PATH
    assert f(None, B, 4, 8, F32, F32, 0, None) == NULL
    assert f(A, None, 4, 8, F32, F32, 0, None) == NULL
    assert f(A + 2, B, 4, 8, F32, F32, 0, None) == ALIGN
    assert f(A, B + 1, 4, 8, F32, BF16, 0, None) == ALIGN
    assert f(A, A + 4, 4, 8, F32, F32, 0, None) == ALIAS          # shifted by one element
    assert f(A, A, 4, 8, F32, BF16, 0, None) == ALIAS             # in place needs one dtype
    assert f(A, A + 4 * 31, 4, 8, F32, F32, 0, None) == ALIAS     # last element shared
    # rows == 0 is a no-op, even with NULL pointers
    assert f(None, None, 0, 8, F32, F32, 0, None) == OK
    assert lib.os_softmax_fwd(None, None, 0, 8, BF16, BF16, None) == OK


def _no_device():
    import torch
    return not torch.cuda.is_available()


# These two pass fake addresses that are only safe because no device exists:
# with a GPU present they would launch on them, so they are skipped there.
@pytest.mark.skipif(not _no_device(), reason="only meaningful (and only safe) without a GPU")
def test_softmax_without_device_fails_loudly(lib):
    # valid arguments but no GPU: the call reports a CUDA error, it never computes on the host
    assert lib.os_softmax_fwd(A, A + 4 * 32, 4, 8, F32, F32, None) == CUDA


@pytest.mark.parametrize("name", ["os_softmax_topk", "os_topk"])
def test_topk_argument_errors(lib, name):
    f = getattr(lib, name)
    assert f(A, B, C, 4, 100, 0, None) == KERR
    assert f(A, B, C, 4, 1000, 257, None) == KERR
    assert f(A, B, C, 4, 5, 6, None) == KERR
    assert f(A, B, C, 4, 0, 1, None) == SHAPE
    assert f(A, B, C, -2, 100, 8, None) == SHAPE
    assert f(None, B, C, 4, 100, 8, None) == NULL
    assert f(A, None, C, 4, 100, 8, None) == NULL
    assert f(A, B, None, 4, 100, 8, None) == NULL
    assert f(A + 1, B, C, 4, 100, 8, None) == ALIGN
    assert f(A, A + 16, C, 4, 100, 8, None) == ALIAS
    assert f(A, B, B + 8, 4, 100, 8, None) == ALIAS
    assert f(None, None, None, 0, 100, 8, None) == OK


def test_stats_argument_errors(lib):
    f = lib.os_softmax_stats
    assert f(A, B, C, C + 4096, 4, 8, 2, None) == DTYPE
    assert f(A, B, C, C + 4096, -1, 8, F32, None) == SHAPE
    assert f(A, B, C, C + 4096, 4, 0, F32, None) == SHAPE
    assert f(None, B, C, C + 4096, 4, 8, F32, None) == NULL
    assert f(A, None, None, None, 4, 8, F32, None) == NULL
    assert f(A + 2, B, C, C + 4096, 4, 8, F32, None) == ALIGN
    assert f(A, A + 16, None, None, 4, 8, F32, None) == ALIAS        # m inside x
    assert f(A, B, B + 8, None, 4, 8, F32, None) == ALIAS            # m and d overlap
    assert f(None, None, None, None, 0, 8, F32, None) == OK


def test_causal_argument_errors(lib):
    f = lib.os_softmax_causal_fwd
    assert f(A, B, 4, 8, 0, 0, F32, F32, None) == SHAPE
    assert f(A, B, 4, 8, 4, -1, F32, F32, None) == SHAPE
    assert f(A, B, 4, 8, 4, 0, 2, F32, None) == DTYPE
    assert f(None, B, 4, 8, 4, 0, F32, F32, None) == NULL
    assert f(A, A + 4, 4, 8, 4, 0, F32, F32, None) == ALIAS
    assert f(A, A, 4, 8, 4, 0, BF16, F32, None) == ALIAS
    assert f(None, None, 0, 8, 4, 0, F32, F32, None) == OK


def test_sample_argument_errors(lib):
    f = lib.os_topk_sample
    D = C + 65536
    assert f(A, B, C, D, -1, 8, None) == SHAPE
    assert f(A, B, C, D, 4, 0, None) == KERR
    assert f(A, B, C, D, 4, 257, None) == KERR
    assert f(None, B, C, D, 4, 8, None) == NULL
    assert f(A, B, C, None, 4, 8, None) == NULL
    assert f(A, B, C + 2, D, 4, 8, None) == ALIGN
    assert f(A, B, C, A + 16, 4, 8, None) == ALIAS
    assert f(None, None, None, None, 0, 8, None) == OK


def test_attention_argument_errors(lib):
    f = lib.os_attention_fwd
    D = 0xC000000  # o; 16-byte aligned, clear of A, B, C for these sizes
    E = 0xE000000  # lse
    s = 0.125
    assert f(A, B, C, D, E, -1, 128, 64, s, 0, None) == SHAPE
    assert f(A, B, C, D, E, 2, -1, 64, s, 0, None) == SHAPE
    assert f(A, B, C, D, E, 2, 128, 96, s, 0, None) == SHAPE
    assert f(A, B, C, D, E, 2, 2 ** 31, 64, s, 0, None) == SHAPE
    assert f(A, B, C, D, E, 2 ** 31, 4096, 64, s, 0, None) == SHAPE
    assert f(A, B, C, D, E, 2, 128, 64, 0.0, 0, None) == VALUE
    assert f(A, B, C, D, E, 2, 128, 64, -s, 0, None) == VALUE
    assert f(A, B, C, D, E, 2, 128, 64, float("inf"), 0, None) == VALUE
    assert f(A, B, C, D, E, 2, 128, 64, float("nan"), 0, None) == VALUE
    assert f(A, B, C, D, E, 2, 128, 64, s, 2, None) == VALUE
    assert f(None, B, C, D, E, 2, 128, 64, s, 0, None) == NULL
    assert f(A, B, C, None, E, 2, 128, 64, s, 0, None) == NULL
    assert f(A + 8, B, C, D, E, 2, 128, 64, s, 0, None) == ALIGN
    assert f(A, B, C, D + 8, E, 2, 128, 64, s, 0, None) == ALIGN
    assert f(A, B, C, D, E + 2, 2, 128, 64, s, 0, None) == ALIGN
    assert f(A, B, C, A + 16, E, 2, 128, 64, s, 0, None) == ALIAS
    assert f(A, B, C, D, D + 64, 2, 128, 64, s, 0, None) == ALIAS
    assert f(A, B, C, D, C, 2, 128, 64, s, 0, None) == ALIAS
    assert f(None, None, None, None, None, 0, 128, 64, s, 0, None) == OK
    assert f(None, None, None, None, None, 4, 0, 128, s, 1, None) == OK


def test_exp_argument_errors(lib):
    assert lib.os_exp_f32(A, B, -1, None) == SHAPE
    assert lib.os_exp_f32(None, B, 5, None) == NULL
    assert lib.os_exp_f32(A + 2, B, 5, None) == ALIGN
    assert lib.os_exp_f32(None, None, 0, None) == OK
    assert lib.os_exp_pairs_f32(A, B, -1, None) == SHAPE
    assert lib.os_exp_pairs_f32(None, B, 5, None) == NULL
    assert lib.os_exp_pairs_f32(A, B + 2, 5, None) == ALIGN
    assert lib.os_exp_pairs_f32(None, None, 0, None) == OK
    assert lib.os_exp_pairs_coarse_f32(A, B, -1, None) == SHAPE
    assert lib.os_exp_pairs_coarse_f32(None, B, 5, None) == NULL
    assert lib.os_exp_pairs_coarse_f32(A, B + 2, 5, None) == ALIGN
    assert lib.os_exp_pairs_coarse_f32(None, None, 0, None) == OK


def test_testing_controls_validate(lib):
    assert lib.os_set_wait_timeout_ns(0) == SHAPE
    assert lib.os_set_wait_timeout_ns(999_999) == SHAPE     # below the 1 ms floor
    assert lib.os_set_wait_timeout_ns(10 ** 6) == OK
    assert lib.os_set_wait_timeout_ns(20 * 10 ** 9) == SHAPE
    assert lib.os_set_wait_timeout_ns(10 ** 9) == OK
    assert lib.os_set_fault_injection(5) == SHAPE
    assert lib.os_set_fault_injection(0) == OK


def test_tensor_helpers_refuse_host_tensors(lib):
    import torch

    import softmax_topk_gb300 as st
    with pytest.raises(ValueError):
        st.softmax(torch.zeros(2, 3))
    with pytest.raises(ValueError):
        st.softmax_topk(torch.zeros(2, 3), 1)


@pytest.mark.skipif(not _no_device(), reason="only meaningful without a GPU")
def test_plan_without_device_reports_cuda_error(lib):
    import softmax_topk_gb300 as st
    with pytest.raises(st.OsError) as e:
        st.os_softmax_plan(4, 1000, F32, F32)
    assert e.value.name == "OS_ERR_CUDA"
