"""The longest row the C ABI accepts (cols = 2^31 - 1), softmax in fp32 and
bf16.  The row's (m, d) comes from the oracle over chunks of the row (each
reshaped into many short rows for its row loop) folded with the oracle's
(+); outputs are checked on samples one by one against e^(x - m) / d, and
the whole row's sum."""
import numpy as np
import pytest
import torch

import oracle
from tests._compare import FLT_MIN, TOL, SUM_TOL

pytestmark = pytest.mark.gpu

MAX_COLS = 2 ** 31 - 1
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _row(dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(1, MAX_COLS, generator=g, device="cuda") * 3.0
    return x.to(DT[dtype]) if dtype != "f32" else x


def _row_stats(x):
    """(m, d) of the single row x[0] by the oracle, chunk by chunk."""
    state = (-np.inf, 0.0)
    chunk, sub = 1 << 26, 1 << 16
    for c0 in range(0, x.shape[1], chunk):
        xc = x[0, c0:c0 + chunk].double().cpu().numpy()
        n = xc.size - xc.size % sub
        parts = [xc[:n].reshape(-1, sub)] + ([xc[n:][None, :]] if n < xc.size else [])
        for part in parts:
            m, d = oracle.row_stats(part)
            for mi, di in zip(m, d):
                state = oracle.combine(state, (float(mi), float(di)))
    return state


def _samples(seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(1000), MAX_COLS - 1 - np.arange(1000),
                                     g.integers(0, MAX_COLS, 2000)]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_longest_row(st, dtype):
    x = _row(dtype, seed=71)
    y = st.softmax(x)
    torch.cuda.synchronize()
    m, d = _row_stats(x)
    at = torch.from_numpy(_samples(5)).cuda()
    xs = x[0, at].double().cpu().numpy()
    ys = y[0, at].double().cpu().numpy()
    ref = np.exp(xs - m) / d
    big = ref >= FLT_MIN
    rel = np.abs(ys[big] - ref[big]) / ref[big]
    assert rel.max() <= TOL[dtype], f"max rel {rel.max():.3e}"
    assert np.all((ys[~big] >= 0) & (ys[~big] <= FLT_MIN))
    total = float(torch.sum(y, dtype=torch.float64))
    assert abs(total - 1.0) <= SUM_TOL[dtype], total
