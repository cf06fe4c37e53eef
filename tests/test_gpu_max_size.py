"""The longest row the C ABI accepts (cols = 2^31 - 1): softmax in fp32 and
bf16, and the fused and plain TopK.  The row's (m, d) comes from the oracle
over chunks of the row (each reshaped into many short rows for its row loop)
folded with the oracle's (+); softmax outputs are checked on samples one by
one against e^(x - m) / d, and the whole row's sum; TopK values against
e^(x - m) / d of the selected columns, indices by the selection rule itself
(nothing outside beats the K-th, ties at it go to the lowest columns).  At
this length each CTA of the row's cluster holds a segment of about 2^28
columns, far more blocks than its candidate list, so the selection takes the
exact path (bisection over the segment's order keys, 64-bit element
indices) -- the part a row of zeros exercises with every column tied."""
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


def test_softmax_topk_longest_row(st):
    x = _row("f32", seed=73)
    x[0, 12345] = 20.0          # a tie at the maximum, at a lower and a higher column
    x[0, MAX_COLS - 7] = 20.0
    K = 8
    vals, idx = st.softmax_topk(x, K)
    torch.cuda.synchronize()
    idx = idx[0].long()
    picked = x[0, idx].double()
    assert idx[0].item() == 12345 and idx[1].item() == MAX_COLS - 7
    assert torch.all(picked[:-1] >= picked[1:])
    vk = float(picked[-1])
    above = int((x[0] > vk).sum())
    at_vk = torch.nonzero(x[0] == vk).flatten()
    assert above < K and above + at_vk.numel() >= K
    need = K - above
    assert torch.equal(idx[above:].sort().values, at_vk[:need])  # ties at the K-th: lowest columns
    m, d = _row_stats(x)
    ref = np.exp(picked.cpu().numpy() - m) / d
    rel = np.abs(vals[0].double().cpu().numpy() - ref) / ref
    assert rel.max() <= TOL["f32"], f"max rel {rel.max():.3e}"


@pytest.mark.parametrize("K", [8, 256])
def test_topk_longest_row_all_tied(st, K):
    """Every column 0 (half of them -0.0): the exact path on every CTA of the
    cluster; the K lowest columns, values 1/cols (fused) or the zeros with
    their own signs (plain)."""
    x = torch.zeros(1, MAX_COLS, device="cuda")
    x[0, 1::2] = -0.0
    vals, idx = st.softmax_topk(x, K)
    pv, pi = st.topk(x, K)
    torch.cuda.synchronize()
    want = torch.arange(K, dtype=torch.int32, device="cuda")
    assert torch.equal(idx[0], want) and torch.equal(pi[0], want)
    rel = (vals[0].double() * MAX_COLS - 1).abs().max()
    assert float(rel) <= TOL["f32"]
    assert torch.equal(pv[0].view(torch.int32), x[0, :K].view(torch.int32))
