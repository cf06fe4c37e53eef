"""Row statistics (m, d, log-sum-exp) and in-kernel causal masking on the GPU,
against the float64 oracle.

m is an input value and must match exactly; d within 1e-5 relative (the
accurate exponential, fp32 accumulation); lse = m + ln d within 2e-6 + 1e-6
|lse| (d's error through the logarithm plus fp32 rounding of the sum).
Causal outputs follow the softmax rule of tests/_compare.py, and masked
entries must be exactly +0.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._compare import assert_softmax_close

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _inputs(rows, cols, dtype, seed, neg_inf_p=0.02):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device="cuda") * 3
    if cols > 2:
        x.masked_fill_(torch.rand(rows, cols, generator=g, device="cuda") < neg_inf_p, -np.inf)
        x[:, seed % cols] = 0.25
    return x.to(DT[dtype])


def _check_stats(st, x, label):
    m, d, lse = st.softmax_stats(x)
    torch.cuda.synchronize()
    x64 = x.double().cpu().numpy()
    rm, rd = oracle.row_stats(x64)
    rl = oracle.lse(x64)
    m, d, lse = (t.double().cpu().numpy() for t in (m, d, lse))
    assert np.array_equal(m, rm), f"{label}: m differs"
    finite = np.isfinite(rm)
    assert np.all(np.abs(d[finite] - rd[finite]) <= 1e-5 * rd[finite]), f"{label}: d"
    assert np.all(np.abs(lse[finite] - rl[finite]) <= 2e-6 + 1e-6 * np.abs(rl[finite])), \
        f"{label}: lse max err {np.abs(lse[finite] - rl[finite]).max():.3e}"
    n_finite = np.isfinite(x64).sum(axis=1)
    assert np.all(d[finite] >= 1.0 - 1e-6) and np.all(d[finite] <= n_finite[finite] * (1 + 1e-6))
    assert np.all(d[~finite] == 0) and np.all(m[~finite] == -np.inf) and np.all(lse[~finite] == -np.inf)


@pytest.mark.parametrize("cols", [1, 2, 7, 64, 100, 1023, 1024, 1025, 4096, 32000, 50257, 131073])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stats_shapes(st, cols, dtype):
    rows = 5 if cols > 100000 else 37
    _check_stats(st, _inputs(rows, cols, dtype, seed=cols + 3), f"{dtype} cols={cols}")


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if w.op == "softmax"])
def test_stats_workload_recipes(st, name):
    w = workloads.WORKLOADS[name]
    rows = min(w.rows, 300 if w.cols <= 4096 else 24)
    _check_stats(st, workloads.make(w.scaled(rows=rows), device="cuda"), name)


def test_stats_edge_rows_and_optional_outputs(st):
    x = torch.randn(6, 3000, device="cuda")
    x[2] = -np.inf
    x[4] = 7.5                                   # constant row: d = n, lse = c + ln n
    _check_stats(st, x, "edge rows")
    lse = torch.empty(6, device="cuda")
    st.os_softmax_stats(x.data_ptr(), None, None, lse.data_ptr(), 6, 3000, st.OS_F32,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert abs(float(lse[4]) - (7.5 + np.log(3000.0))) <= 1e-5
    with pytest.raises(st.OsError) as e:
        st.os_softmax_stats(x.data_ptr(), None, None, None, 6, 3000, st.OS_F32, None)
    assert e.value.name == "OS_ERR_NULL"


def test_stats_agree_with_softmax_output(st):
    """softmax = e^(x - m) / d with the exported (m, d)."""
    x = _inputs(16, 20000, "f32", seed=9)
    m, d, _ = st.softmax_stats(x)
    y = st.softmax(x)
    y2 = torch.exp(x.double() - m.double()[:, None]) / d.double()[:, None]
    rel = ((y.double() - y2).abs() / y2.clamp_min(1e-30))[y2 > 1e-30].max()
    assert float(rel) <= 2e-5


CAUSAL = [  # rows, cols, period, offset: warp rows, stream rows, offsets past the end
    (384, 128, 128, 0), (100, 33, 7, 0), (64, 1000, 64, 900), (48, 4096, 16, 4000),
    (40, 50257, 40, 50000), (12, 131073, 6, 131000), (20, 300, 5, 1000),
    # at least as many rows as SMs, rows of up to 96 KB: 256-thread streaming CTAs
    (160, 4097, 160, 3000), (200, 24576, 50, 24500), (160, 12001, 160, 11900)]


@pytest.mark.parametrize("rows,cols,period,offset", CAUSAL)
@pytest.mark.parametrize("pair", [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16")],
                         ids=lambda p: f"{p[0]}-{p[1]}")
def test_causal_matches_oracle(st, rows, cols, period, offset, pair):
    x = _inputs(rows, cols, pair[0], seed=cols + period)
    y = st.softmax_causal(x, period, offset, out_dtype=DT[pair[1]])
    torch.cuda.synchronize()
    x64 = x.double().cpu().numpy()
    ref = oracle.softmax_causal(x64, period, offset)
    masked = oracle.causal_mask(x64, period, offset)
    yy = y.double().cpu().numpy()
    assert_softmax_close(masked, yy, ref, pair[1], f"causal {rows}x{cols} p={period} o={offset}")
    keep = np.arange(cols)[None, :] <= (np.arange(rows)[:, None] % period) + offset
    assert np.all(yy[~keep] == 0.0) and not np.any(np.signbit(yy[~keep]))


def test_causal_workload_equals_reading_minus_inf(st):
    """The causal recipe (1048576 x 128, -inf planted above the diagonal) and the
    same rows without the planted -inf under the in-kernel mask give the same
    probabilities."""
    w = workloads.WORKLOADS["causal_1048576x128_f32"]
    x = workloads.make(w.scaled(rows=4096), device="cuda")
    dense = torch.where(torch.isinf(x), torch.zeros_like(x), x)
    y_read = st.softmax(x)
    y_mask = st.softmax_causal(dense, 128, 0)
    torch.cuda.synchronize()
    rel = ((y_read.double() - y_mask.double()).abs() / y_read.double().clamp_min(1e-30))
    assert float(rel[y_read > 0].max()) <= 1e-6 and torch.all(y_mask[y_read == 0] == 0)


def test_causal_argument_errors(st):
    x = torch.randn(4, 64, device="cuda")
    y = torch.empty_like(x)
    for period, offset in ((0, 0), (-3, 0), (4, -1)):
        with pytest.raises(st.OsError) as e:
            st.os_softmax_causal_fwd(x.data_ptr(), y.data_ptr(), 4, 64, period, offset,
                                     st.OS_F32, st.OS_F32, None)
        assert e.value.name == "OS_ERR_SHAPE"


def test_stats_outputs_do_not_touch_neighbours(st):
    """m, d and lse written into the middle of guard-filled buffers (warp and
    CTA families): the guard bands stay untouched."""
    G = 512
    for rows, cols, dtype in ((300, 700, "f32"), (50, 40000, "bf16")):
        x = _inputs(rows, cols, dtype, seed=cols)
        bufs = [torch.full((rows + 2 * G,), 3.5, device="cuda") for _ in range(3)]
        m, d, lse = (b[G:G + rows] for b in bufs)
        st.os_softmax_stats(x.data_ptr(), m.data_ptr(), d.data_ptr(), lse.data_ptr(), rows, cols,
                            st.OS_F32 if dtype == "f32" else st.OS_BF16,
                            torch.cuda.current_stream().cuda_stream)
        rm, rd, rl = st.softmax_stats(x)
        torch.cuda.synchronize()
        for b in bufs:
            assert torch.all(b[:G] == 3.5) and torch.all(b[G + rows:] == 3.5)
        assert torch.equal(m, rm) and torch.equal(d, rd) and torch.equal(lse, rl)
