"""Fused softmax+TopK parity on the GPU against the float64 oracle.

Indices must match bit for bit (ties go to the lower column index); values
within 1e-5 relative (values below FLT_MIN: in [0, FLT_MIN]).  Shapes cross
the tile and cluster capacities, rows start at every 4-byte offset inside a
16-byte vector, and crafted inputs drive the candidate-overflow path.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._compare import assert_topk_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _run(st, x, K, label):
    vals, idx = st.softmax_topk(x, K)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(x.double().cpu().numpy(), K)
    assert_topk_equal(vals.cpu().numpy(), idx.cpu().numpy(), rv, ri, label)


def _rand(rows, cols, seed, scale=4.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(rows, cols, generator=g, device="cuda") * scale


COLS = [1, 2, 3, 5, 8, 63, 64, 65, 100, 1000, 4097, 8191, 8192, 8193, 16387, 32771, 50257,
        65539, 100003, 300007]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("K", [1, 2, 7, 8, 33, 64, 65, 100, 256])
def test_shapes(st, cols, K):
    if K > cols:
        pytest.skip("K > cols")
    rows = 3 if cols > 100000 else 9     # 9 rows: every start offset mod 16 bytes occurs
    _run(st, _rand(rows, cols, seed=cols * 131 + K), K, f"cols={cols} K={K}")


@pytest.mark.parametrize("K", [8, 64, 256])
def test_workload_full_size(st, K):
    w = workloads.WORKLOADS["topk_256x50257_f32"]
    x = workloads.make(w, device="cuda")
    _run(st, x, K, f"{w.name} K={K}")


@pytest.mark.parametrize("K", [8, 64, 200])
def test_workload_with_planted_ties(st, K):
    w = workloads.WORKLOADS["topk_256x50257_f32"]
    x = workloads.plant_ties(workloads.make(w.scaled(rows=64), device="cuda"), per_row=K // 2 + 3)
    _run(st, x, K, f"ties K={K}")


@pytest.mark.parametrize("cols", [100, 5000, 50257])
def test_coarse_values_many_ties(st, cols):
    g = torch.Generator(device="cuda")
    g.manual_seed(cols)
    x = torch.randint(0, 4, (6, cols), generator=g, device="cuda").float()
    for K in (1, 8, 64, 256):
        if K <= cols:
            _run(st, x, K, f"values in 0..3, cols={cols} K={K}")


@pytest.mark.parametrize("cols", [70, 9000, 50257, 200000])
def test_constant_rows_overflow_path(st, cols):
    """Every entry ties: the threshold admits far more than the candidate
    buffer holds, so the kernel merges in several passes."""
    x = torch.full((3, cols), 2.5, device="cuda")
    for K in (8, 64, 256):
        if K <= cols:
            _run(st, x, K, f"constant cols={cols} K={K}")


def test_fewer_finite_than_k(st):
    x = torch.full((4, 5000), -np.inf, device="cuda")
    x[0, 4999] = 1.0
    x[1, [0, 17, 4000]] = torch.tensor([0.5, 0.5, -2.0], device="cuda")
    x[2, 100:110] = torch.arange(10, dtype=torch.float32, device="cuda")
    x[3, 1] = 3.0
    _run(st, x, 64, "few finite entries")
    _run(st, x, 256, "few finite entries, K = 256")


def test_increasing_and_decreasing_rows(st):
    up = torch.arange(60000, dtype=torch.float32, device="cuda")[None, :] * 1e-3
    x = torch.cat([up, up.flip(1), -up]).contiguous()
    for K in (8, 64, 256):
        _run(st, x, K, f"monotone K={K}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_base(st, offset):
    rows, cols, K = 5, 50257, 64
    buf = torch.empty(rows * cols + 8, device="cuda")
    x = buf[offset:offset + rows * cols].view(rows, cols)
    x.copy_(_rand(rows, cols, seed=offset))
    vals = torch.empty(rows, K, device="cuda")
    idx = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    st.os_softmax_topk(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, cols, K,
                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(x.double().cpu().numpy(), K)
    assert_topk_equal(vals.cpu().numpy(), idx.cpu().numpy(), rv, ri, f"offset {offset}")


def test_many_rows_short(st):
    _run(st, _rand(5000, 40, seed=3), 16, "5000 x 40")


MANY_ROWS = 640  # at least four CTAs of 256 threads per SM


@pytest.mark.parametrize("cols", [1000, 8193, 32000, 50257, 65536, 65537])
@pytest.mark.parametrize("K", [1, 8, 64])
def test_many_row_batches(st, cols, K):
    """Batches of at least as many rows as resident 256-thread CTAs run the
    256-thread build (rows of up to 65536 columns, K <= 64); fused and plain,
    with ties planted at each row's maximum in half the rows."""
    rows = MANY_ROWS
    plan = st.os_topk_plan(rows, cols, K)
    assert plan["cluster"] == 1 and plan["threads"] == (256 if cols <= 65536 else 512), plan
    x = _rand(rows, cols, seed=cols + K)
    top = x.max(dim=1, keepdim=True).values
    g = torch.Generator(device="cuda")
    g.manual_seed(cols * 7 + K)
    pos = torch.randint(0, cols, (rows // 2, 5), generator=g, device="cuda")
    x[: rows // 2].scatter_(1, pos, top[: rows // 2].expand(-1, 5))
    _run(st, x, K, f"{rows}x{cols} K={K}")
    _run_plain(st, x, K, f"plain {rows}x{cols} K={K}")


@pytest.mark.parametrize("offset", [1, 3])
def test_many_row_batches_misaligned(st, offset):
    rows, cols, K = MANY_ROWS, 20011, 64
    buf = torch.empty(rows * cols + 8, device="cuda")
    x = buf[offset:offset + rows * cols].view(rows, cols)
    x.copy_(_rand(rows, cols, seed=offset + 5))
    assert st.os_topk_plan(rows, cols, K)["threads"] == 256
    vals = torch.empty(rows, K, device="cuda")
    idx = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    st.os_softmax_topk(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, cols, K,
                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(x.double().cpu().numpy(), K)
    assert_topk_equal(vals.cpu().numpy(), idx.cpu().numpy(), rv, ri, f"{rows} rows offset {offset}")


def test_values_equal_softmax_output(st):
    x = _rand(16, 32000, seed=11)
    vals, idx = st.softmax_topk(x, 64)
    y = st.softmax(x)
    picked = torch.gather(y, 1, idx.long())
    rel = ((picked.double() - vals.double()).abs() / vals.double()).max()
    assert float(rel) <= 2e-5


def test_bad_k_raises(st):
    x = _rand(2, 100, seed=1)
    with pytest.raises(st.OsError) as e:
        st.softmax_topk(_rand(2, 1000, seed=1), 257)
    assert e.value.name == "OS_ERR_K"
    with pytest.raises(st.OsError):
        st.softmax_topk(_rand(2, 10, seed=1), 11)


# ------------------------------------------------------------------ os_topk (TopK of x itself)
def _run_plain(st, x, K, label):
    vals, idx = st.topk(x, K)
    torch.cuda.synchronize()
    x64 = x.double().cpu().numpy()
    _, ri = oracle.topk(x64, K)  # the oracle's order: value descending, then column ascending
    idx = idx.cpu().numpy()
    bad = np.argwhere(idx != ri)
    assert bad.size == 0, f"{label}: {len(bad)} index mismatches, first at {bad[:3].tolist()}"
    want = np.take_along_axis(x.cpu().numpy(), idx.astype(np.int64), axis=1)
    assert np.array_equal(vals.cpu().numpy(), want), f"{label}: values are not the selected x"


@pytest.mark.parametrize("cols", [1, 5, 64, 65, 1000, 8193, 50257, 300007])
@pytest.mark.parametrize("K", [1, 8, 64, 256])
def test_plain_topk_shapes(st, cols, K):
    if K > cols:
        pytest.skip("K > cols")
    rows = 3 if cols > 100000 else 9
    _run_plain(st, _rand(rows, cols, seed=cols * 7 + K), K, f"plain cols={cols} K={K}")


def test_plain_topk_ties_and_inf(st):
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randint(0, 4, (6, 20000), generator=g, device="cuda").float()
    x[1] = -np.inf
    x[1, [3, 19999]] = 0.0
    for K in (1, 8, 64):
        _run_plain(st, x, K, f"plain ties K={K}")


@pytest.mark.parametrize("K", [8, 64, 200, 256])
def test_sorted_selection_zero_ties(st, K):
    """More candidates than the counting rank takes (the radix cut for K <= 64,
    the sort above): rows of -|x| with 600 zeros, half of them -0.0, so the K
    best are all zeros, tied at the K-th key, and must be the lowest columns,
    in column order, with their own sign bits."""
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    rows, cols = 4, 20000
    x = -torch.randn(rows, cols, generator=g, device="cuda").abs() - 1e-3
    for r in range(rows):
        pos = torch.randperm(cols, generator=g, device="cuda")[:600]
        x[r, pos[:300]] = 0.0
        x[r, pos[300:]] = -0.0
    _run_plain(st, x, K, f"zero ties K={K}")
    vals, idx = st.topk(x, K)
    want = torch.gather(x, 1, idx.long())
    assert torch.equal(vals.view(torch.int32), want.view(torch.int32)), "sign of zero lost"
    fv, fi = st.softmax_topk(x, K)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(x.double().cpu().numpy(), K)
    assert_topk_equal(fv.cpu().numpy(), fi.cpu().numpy(), rv, ri, f"fused zero ties K={K}")


def _signed_zero_rows(rows, cols, seed, zeros=None):
    """Rows of zeros with random signs (zeros=None), or rows of negative
    values holding `zeros` random-sign zeros at random columns."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if zeros is None:
        sign = torch.randint(0, 2, (rows, cols), generator=g, device="cuda").bool()
        return torch.where(sign, torch.tensor(-0.0, device="cuda"), torch.tensor(0.0, device="cuda"))
    x = -torch.randn(rows, cols, generator=g, device="cuda").abs() - 1e-3
    for r in range(rows):
        pos = torch.randperm(cols, generator=g, device="cuda")[:zeros]
        half = zeros // 2
        x[r, pos[:half]] = 0.0
        x[r, pos[half:]] = -0.0
    return x


def _check_fused_and_plain(st, x, K, label):
    _run(st, x, K, f"fused {label}")
    _run_plain(st, x, K, f"plain {label}")
    vals, idx = st.topk(x, K)
    want = torch.gather(x, 1, idx.long())
    assert torch.equal(vals.view(torch.int32), want.view(torch.int32)), f"sign of zero lost: {label}"


# (rows, cols): 320 rows run one CTA per row; 16 rows of 50257 split each row
# over a cluster; 640 rows run CTAs of 256 threads for K <= 64; 5000 and 7003
# columns with more than 2048 zeros overflow the candidate buffer, so the row
# takes the exact path
@pytest.mark.parametrize("shape", [(320, 5000), (16, 50257), (7, 7003), (640, 5000)])
@pytest.mark.parametrize("K", [8, 64, 256])
def test_exact_path_signed_zero_ties(st, shape, K):
    """More than 2048 candidates tied at zero, half of them -0.0: the exact
    path must rank -0 and +0 as one value and take the lowest columns, fused
    and plain, one CTA per row and clusters; plain values keep their signs."""
    rows, cols = shape
    plan = st.os_topk_plan(rows, cols, K)
    x = _signed_zero_rows(rows, cols, seed=rows + cols + K)
    _check_fused_and_plain(st, x, K, f"all zeros {rows}x{cols} K={K} S={plan['cluster']}")
    x = _signed_zero_rows(rows, cols, seed=rows * cols + K, zeros=min(cols - 1, 4000))
    _check_fused_and_plain(st, x, K, f"4000 zeros {rows}x{cols} K={K} S={plan['cluster']}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_exact_path_misaligned_ragged(st, offset):
    """The exact path on rows that start inside a 16-byte block and end in a
    partial block (4-byte offsets, odd row length), through the raw C entry
    points, fused and plain."""
    rows, cols, K = 5, 6001, 64
    buf = torch.empty(rows * cols + 8, device="cuda")
    x = buf[offset:offset + rows * cols].view(rows, cols)
    x.copy_(_signed_zero_rows(rows, cols, seed=offset * 11))
    rv, ri = oracle.topk(x.double().cpu().numpy(), K)
    for fn in (st.os_softmax_topk, st.os_topk):
        vals = torch.empty(rows, K, device="cuda")
        idx = torch.empty(rows, K, dtype=torch.int32, device="cuda")
        fn(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, cols, K,
           torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ri), f"offset {offset} {fn.__name__}"
        if fn is st.os_softmax_topk:
            assert_topk_equal(vals.cpu().numpy(), idx.cpu().numpy(), rv, ri, f"offset {offset}")
        else:
            want = torch.gather(x, 1, idx.long())
            assert torch.equal(vals.view(torch.int32), want.view(torch.int32))


@pytest.mark.parametrize("K", [8, 64])
def test_unfused_pipeline_matches_fused(st, K):
    """softmax then TopK of the probabilities (the unfused pipeline) against the
    oracle's TopK of those probabilities, and against the fused kernel's values."""
    w = workloads.WORKLOADS["topk_256x50257_f32"]
    x = workloads.make(w.scaled(rows=32), device="cuda")
    y = st.softmax(x)
    _run_plain(st, y, K, f"TopK of softmax(x) K={K}")
    vals_u, _ = st.topk(y, K)
    vals_f, _ = st.softmax_topk(x, K)
    rel = ((vals_u.double() - vals_f.double()).abs() / vals_f.double()).max()
    assert float(rel) <= 2e-5


# ------------------------------------------------------------------ top-K sampling
def _sample_window(vals, u):
    """The fp32 rounding window of each row's draw: the kernel rounds each of
    its K partial sums and the product u * total to fp32, so every compared
    quantity is within (K + 1) 2^-24 of the total of its exact value (all
    values are >= 0).  Returns the exact partial sums, the exact targets and
    the window half-width per row."""
    v = vals.astype(np.float64)
    K = v.shape[1]
    total = v.sum(axis=1)
    return np.cumsum(v, axis=1), u * total, 2 * (K + 1) * 2.0 ** -24 * total


@pytest.mark.parametrize("K", [1, 8, 64, 256])
def test_topk_sample_matches_oracle(st, K):
    """Fused TopK, then one draw per row; the float64 oracle draws from the
    same (value, index) pairs and the same u.  Every row whose target is not
    within fp32 rounding of a cumulative-sum boundary must agree exactly;
    on the (few, counted) ambiguous rows the kernel's pick must be a position
    the rounding window allows: its partial sum reaches the target and the
    one before does not, each up to the window."""
    w = workloads.WORKLOADS["topk_256x50257_f32"]
    x = workloads.make(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(100 + K)
    u = torch.rand(w.rows, generator=g, device="cuda")
    samples, vals, idx = st.softmax_topk_sample(x, K, u)
    torch.cuda.synchronize()
    v, ix, uu = vals.double().cpu().numpy(), idx.cpu().numpy(), u.double().cpu().numpy()
    got = samples.cpu().numpy()
    want = oracle.topk_sample(v, ix, uu)
    run, target, win = _sample_window(v, uu)
    amb = np.abs(run - target[:, None]).min(axis=1) <= win
    assert np.array_equal(got[~amb], want[~amb]), \
        f"K={K}: {int((got[~amb] != want[~amb]).sum())} unambiguous rows differ"
    for r in np.nonzero(amb)[0]:
        k = int(np.nonzero(ix[r] == got[r])[0][0])
        below = run[r, k - 1] if k > 0 else 0.0
        assert below <= target[r] + win[r], (r, k)
        assert k == K - 1 or run[r, k] > target[r] - win[r], (r, k)
    print(f"K={K}: {int(amb.sum())} of {w.rows} rows within fp32 rounding of a boundary, "
          f"{int((got[amb] != want[amb]).sum())} of them drawn differently")
    assert np.all(np.any(ix == got[:, None], axis=1))


def test_topk_sample_near_boundaries(st):
    """Non-dyadic values with u placed a clear margin (1e-5 of the total) on
    either side of each cumulative-sum boundary: the float64 oracle and the
    fp32 kernel must pick the same entry."""
    p = np.array([0.1, 0.2, 0.3, 0.4], dtype=np.float32)
    bounds = np.cumsum(p.astype(np.float64))[:-1] / p.astype(np.float64).sum()
    us = np.concatenate([bounds - 1e-5, bounds + 1e-5]).astype(np.float32)
    rows = len(us)
    vals = torch.tensor(np.tile(p, (rows, 1)), device="cuda")
    idx = (torch.arange(4, dtype=torch.int32, device="cuda") + 20).repeat(rows, 1).contiguous()
    u = torch.tensor(us, device="cuda")
    out = st.topk_sample(vals, idx, u).cpu().numpy()
    want = oracle.topk_sample(np.tile(p.astype(np.float64), (rows, 1)), idx.cpu().numpy(),
                              us.astype(np.float64))
    assert np.array_equal(out, want)
    assert list(out) == [20, 21, 22, 21, 22, 23]


def test_topk_sample_frequencies(st):
    rows, K = 4096, 4
    vals = torch.tensor([[0.5, 0.25, 0.125, 0.125]], device="cuda").repeat(rows, 1)
    idx = (torch.arange(K, dtype=torch.int32, device="cuda") + 3).repeat(rows, 1).contiguous()
    u = ((torch.arange(rows, device="cuda", dtype=torch.float64) + 0.5) / rows).float()
    out = st.topk_sample(vals, idx, u)
    counts = torch.bincount(out.long() - 3, minlength=K)
    assert counts.tolist() == [2048, 1024, 512, 512]
    edge = st.topk_sample(torch.tensor([[0.0, 0.3, 0.7]] * 2, device="cuda"),
                          torch.tensor([[5, 6, 7]] * 2, dtype=torch.int32, device="cuda"),
                          torch.tensor([0.0, 1.0], device="cuda"))
    assert edge.tolist() == [6, 7]


@pytest.mark.parametrize("K", [8, 64, 256])
def test_outputs_do_not_touch_neighbours(st, K):
    """vals and idx written into the middle of guard-filled buffers (fused
    and plain TopK, several rows per CTA and clusters), then the sampler's
    output likewise: the guard bands stay untouched and the results match
    a run into fresh buffers."""
    G = 1024
    for rows, cols in ((3, 300007), (40, 50257), (700, 3001)):
        x = _rand(rows, cols, seed=rows * 7 + K)
        for fn in (st.os_softmax_topk, st.os_topk):
            vb = torch.full((rows * K + 2 * G,), 7.0, device="cuda")
            ib = torch.full((rows * K + 2 * G,), -5, dtype=torch.int32, device="cuda")
            vals, idx = vb[G:G + rows * K], ib[G:G + rows * K]
            fn(x.data_ptr(), vals.data_ptr(), idx.data_ptr(), rows, cols, K,
               torch.cuda.current_stream().cuda_stream)
            ref_v, ref_i = (st.softmax_topk(x, K) if fn is st.os_softmax_topk else st.topk(x, K))
            torch.cuda.synchronize()
            assert torch.all(vb[:G] == 7.0) and torch.all(vb[G + rows * K:] == 7.0)
            assert torch.all(ib[:G] == -5) and torch.all(ib[G + rows * K:] == -5)
            assert torch.equal(vals.view(rows, K), ref_v) and torch.equal(idx.view(rows, K), ref_i)
        vals, idx = st.softmax_topk(x, K)
        u = torch.rand(rows, device="cuda")
        ob = torch.full((rows + 2 * G,), -9, dtype=torch.int32, device="cuda")
        out = ob[G:G + rows]
        st.topk_sample(vals, idx, u, out=out)
        torch.cuda.synchronize()
        assert torch.all(ob[:G] == -9) and torch.all(ob[G + rows:] == -9)
        assert torch.equal(out, st.topk_sample(vals, idx, u))
