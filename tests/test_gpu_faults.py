"""Bounded device-side waits: data that never arrives (injected on the host: in
the softmax ring kernel the first CTA skips its first bulk copy, in the fused
TopK one CTA of a cluster never sends its list) makes the wait run out after the
configured time; the kernel finishes, the status call reports OS_ERR_TIMEOUT,
and the context stays usable for correct work afterwards.  Nothing traps or
hangs."""
import time

import numpy as np
import pytest
import torch

import oracle
from tests._compare import assert_softmax_close, assert_topk_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    yield softmax_topk_gb300
    softmax_topk_gb300.os_set_fault_injection(0)
    softmax_topk_gb300.os_set_wait_timeout_ns(10 ** 9)


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("shape,dtype", [((64, 32000), torch.float32),
                                         ((32, 128256), torch.bfloat16)])
def test_softmax_wait_times_out_and_recovers(st, shape, dtype):
    x = (torch.randn(*shape, device="cuda") * 2).to(dtype)
    code = st.OS_F32 if dtype == torch.float32 else st.OS_BF16
    assert st.plan(shape, code, path="onchip")["stages"] > 0     # the bulk-copy ring kernel
    st.os_device_status(_stream())                      # clean slate
    st.os_set_wait_timeout_ns(20 * 10 ** 6)             # 20 ms
    st.os_set_fault_injection(1)
    try:
        t0 = time.time()
        st.softmax(x, path="onchip")                    # launch itself succeeds
        with pytest.raises(st.OsError) as e:
            st.os_device_status(_stream())
        assert e.value.name == "OS_ERR_TIMEOUT"
        assert time.time() - t0 < 10.0
    finally:
        st.os_set_fault_injection(0)
        st.os_set_wait_timeout_ns(10 ** 9)
    y = st.softmax(x, path="onchip")
    st.os_device_status(_stream())                      # no error now
    xx = x.double().cpu().numpy()
    out = "f32" if dtype == torch.float32 else "bf16"
    assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), out, "after recovery")


def test_topk_wait_times_out_and_recovers(st):
    x = torch.randn(16, 50257, device="cuda") * 4
    assert st.os_topk_plan(16, 50257, 8)["cluster"] > 1    # rows split over a cluster
    st.os_device_status(_stream())
    st.os_set_wait_timeout_ns(20 * 10 ** 6)
    st.os_set_fault_injection(1)
    try:
        st.softmax_topk(x, 8)
        with pytest.raises(st.OsError) as e:
            st.os_device_status(_stream())
        assert e.value.name == "OS_ERR_TIMEOUT"
    finally:
        st.os_set_fault_injection(0)
        st.os_set_wait_timeout_ns(10 ** 9)
    vals, idx = st.softmax_topk(x, 8)
    st.os_device_status(_stream())
    rv, ri = oracle.topk(x.double().cpu().numpy(), 8)
    assert_topk_equal(vals.cpu().numpy(), idx.cpu().numpy(), rv, ri, "after recovery")


def test_status_clean_after_normal_work(st):
    x = torch.randn(8, 40000, device="cuda")
    st.softmax(x)
    st.softmax_topk(x, 64)
    st.os_device_status(_stream())


def test_timeout_on_one_stream_reported_on_another(st):
    """The status word is read and cleared in one atomic exchange on the
    stream of the call: a wait that gave up in a kernel on a side stream is
    reported by a call on the default stream (once that kernel has finished),
    and the next call finds the word clear."""
    x = (torch.randn(64, 32000, device="cuda") * 2)
    st.os_device_status(_stream())
    side = torch.cuda.Stream()
    st.os_set_wait_timeout_ns(20 * 10 ** 6)
    st.os_set_fault_injection(1)
    try:
        with torch.cuda.stream(side):
            st.softmax(x, path="onchip")
        side.synchronize()
    finally:
        st.os_set_fault_injection(0)
        st.os_set_wait_timeout_ns(10 ** 9)
    with pytest.raises(st.OsError) as e:
        st.os_device_status(_stream())
    assert e.value.name == "OS_ERR_TIMEOUT"
    st.os_device_status(_stream())  # cleared by the exchange
