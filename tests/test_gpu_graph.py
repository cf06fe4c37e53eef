"""The library's calls inside a captured CUDA graph (serving loops replay
one): replays on new inputs give the same bits as direct calls, for every
softmax family the shapes reach, the fused and plain TopK, sampling and the
row statistics; a first use of a kernel may itself happen during capture."""
import numpy as np
import pytest
import torch

import oracle
from tests._compare import assert_softmax_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _randn(shape, seed, dtype=torch.float32, scale=3.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device="cuda") * scale).to(dtype)


# (rows, cols, dtype): warp, on-chip, 256- and 512-thread streaming CTAs, clusters
SHAPES = [(1000, 700, torch.float32), (300, 4096, torch.bfloat16), (400, 20000, torch.float32),
          (320, 50257, torch.bfloat16), (16, 100000, torch.float32)]


@pytest.mark.parametrize("rows,cols,dtype", SHAPES, ids=lambda v: str(v))
def test_softmax_replay_matches_direct_calls(st, rows, cols, dtype):
    x = _randn((rows, cols), seed=cols, dtype=dtype)
    y = torch.empty_like(x)
    st.softmax(x, out=y)  # first use outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.softmax(x, out=y)
        st.softmax(y, out=y)  # in place, chained
    for seed in (1, 2):
        x.copy_(_randn((rows, cols), seed=seed * 1000 + cols, dtype=dtype))
        g.replay()
        torch.cuda.synchronize()
        want = st.softmax(st.softmax(x))
        torch.cuda.synchronize()
        assert torch.equal(y, want), f"replay {seed} differs {rows}x{cols} {dtype}"


def test_first_use_inside_capture(st):
    """A shape and dtype pair not launched before: the kernel's set-up runs
    during the capture."""
    x = _randn((500, 3001), seed=7, dtype=torch.bfloat16)
    y = torch.empty(500, 3001, dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.softmax(x, out_dtype=torch.float32, out=y)
    g.replay()
    torch.cuda.synchronize()
    xx = x.double().cpu().numpy()
    assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), "f32", "captured first use")


@pytest.mark.parametrize("rows,cols,K", [(256, 50257, 8), (700, 32000, 64), (16, 128256, 64),
                                         (64, 5000, 200)])
def test_topk_sampling_replay(st, rows, cols, K):
    x = _randn((rows, cols), seed=rows + K, scale=4.0)
    vals = torch.empty(rows, K, device="cuda")
    idx = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    pv = torch.empty(rows, K, device="cuda")
    pi = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    u = torch.rand(rows, device="cuda")
    draws = torch.empty(rows, dtype=torch.int32, device="cuda")
    st.softmax_topk(x, K, vals=vals, idx=idx)
    st.topk(x, K, vals=pv, idx=pi)
    st.topk_sample(vals, idx, u, out=draws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.softmax_topk(x, K, vals=vals, idx=idx)
        st.topk(x, K, vals=pv, idx=pi)
        st.topk_sample(vals, idx, u, out=draws)
    for seed in (3, 4):
        x.copy_(_randn((rows, cols), seed=seed * 77 + cols, scale=4.0))
        u.copy_(torch.rand(rows, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        v2, i2 = st.softmax_topk(x, K)
        p2, q2 = st.topk(x, K)
        d2 = st.topk_sample(v2, i2, u)
        torch.cuda.synchronize()
        assert torch.equal(vals, v2) and torch.equal(idx, i2), f"fused {rows}x{cols} K={K}"
        assert torch.equal(pv, p2) and torch.equal(pi, q2), f"plain {rows}x{cols} K={K}"
        assert torch.equal(draws, d2), f"sample {rows}x{cols} K={K}"
        _, ri = oracle.topk(x.double().cpu().numpy(), K)
        assert np.array_equal(idx.cpu().numpy(), ri)


def test_stats_and_causal_replay(st):
    x = _randn((2048, 4096), seed=11)
    m = torch.empty(2048, device="cuda")
    d = torch.empty(2048, device="cuda")
    lse = torch.empty(2048, device="cuda")
    y = torch.empty_like(x)
    st.softmax_stats(x, m=m, d=d, lse=lse)
    st.softmax_causal(x, 1024, 100, out=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.softmax_stats(x, m=m, d=d, lse=lse)
        st.softmax_causal(x, 1024, 100, out=y)
    x.copy_(_randn((2048, 4096), seed=12))
    g.replay()
    torch.cuda.synchronize()
    m2, d2, l2 = st.softmax_stats(x)
    y2 = st.softmax_causal(x, 1024, 100)
    torch.cuda.synchronize()
    assert torch.equal(m, m2) and torch.equal(d, d2) and torch.equal(lse, l2)
    assert torch.equal(y, y2)
