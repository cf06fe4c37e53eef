"""Softmax parity on the GPU: every kernel family against the float64 oracle.

Small shapes sweep the column counts that cross every dispatch boundary and
ragged tail (vector width, warp, CTA and cluster capacities); the workload
recipes run scaled down and at full size, every row against the oracle,
plus properties checked on every row.  Tolerances: fp32 output 1e-5 relative,
bf16 output 8e-3 relative (tests/_compare.py states the full rule).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._compare import FLT_MIN, SUM_TOL, assert_softmax_close

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16"), ("bf16", "f32")]
PATHS = ["auto", "warp", "onchip", "stream", "safe", "stream_poly"]
COLS = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256,
        257, 511, 512, 513, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097, 8191, 8192,
        8193, 16383, 16384, 16385, 32000, 32768, 32769, 50257, 65535, 65536, 65537, 128256,
        131072, 131073, 262144, 262145, 524288, 524289]


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _inputs(rows, cols, dtype, seed, scale=3.0, neg_inf_p=0.02):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device="cuda") * scale
    if cols > 2:
        x.masked_fill_(torch.rand(rows, cols, generator=g, device="cuda") < neg_inf_p, -np.inf)
        x[:, (seed * 7919) % cols] = 0.5  # at least one finite entry per row
    return x.to(DT[dtype])


def _check(st, x, out, path, label):
    try:
        y = st.softmax(x, out_dtype=DT[out], path=path)
    except st.OsError as e:
        if e.name == "OS_ERR_PATH":
            pytest.skip(f"{path} cannot hold {tuple(x.shape)}")
        raise
    torch.cuda.synchronize()
    x64 = x.double().cpu().numpy()
    ref = oracle.softmax(x64)
    return assert_softmax_close(x64, y.double().cpu().numpy(), ref, out, label)


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
def test_cols_sweep_auto(st, cols, pair):
    rows = 3 if cols > 100000 else 5
    x = _inputs(rows, cols, pair[0], seed=cols)
    _check(st, x, pair[1], "auto", f"auto {pair} cols={cols}")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("path", ["warp", "onchip", "stream", "safe", "stream_poly"])
@pytest.mark.parametrize("pair", [("f32", "f32"), ("bf16", "bf16")], ids=lambda p: f"{p[0]}-{p[1]}")
def test_cols_sweep_forced_path(st, cols, path, pair):
    rows = 3 if cols > 100000 else 6
    x = _inputs(rows, cols, pair[0], seed=cols + 17)
    _check(st, x, pair[1], path, f"{path} {pair} cols={cols}")


@pytest.mark.parametrize("cols", [7, 64, 1000, 4097, 8193, 32000, 50257, 131073, 262145])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place_matches_out_of_place(st, cols, path, dt):
    """y == x with one dtype: the input is overwritten with exactly the bits
    the same kernel writes to a separate output."""
    rows = 3 if cols > 100000 else 9
    x = _inputs(rows, cols, dt, seed=cols + 29)
    try:
        ref = st.softmax(x, path=path)
    except st.OsError as e:
        if e.name == "OS_ERR_PATH":
            pytest.skip(f"{path} cannot hold {tuple(x.shape)}")
        raise
    z = x.clone()
    y = st.softmax(z, path=path, out=z)
    torch.cuda.synchronize()
    assert y.data_ptr() == z.data_ptr()
    assert torch.equal(z, ref), f"in place differs: {path} {dt} cols={cols}"


@pytest.mark.parametrize("cols", [100, 3001, 32000, 131073])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place_unaligned_rows(st, cols, dt):
    """In place on a buffer that starts one element past a 16-byte boundary
    (rows filled element by element), every path that holds the shape."""
    rows = 5
    src = _inputs(rows, cols, dt, seed=cols + 37)
    for path in PATHS:
        buf = torch.zeros(rows * cols + 8, dtype=src.dtype, device="cuda")
        x = buf[1:1 + rows * cols].view(rows, cols)
        x.copy_(src)
        try:
            ref = st.softmax(x, path=path)
        except st.OsError as e:
            if e.name == "OS_ERR_PATH":
                continue
            raise
        st.softmax(x, path=path, out=x)
        torch.cuda.synchronize()
        assert torch.equal(x, ref), f"in place differs: {path} {dt} cols={cols} (unaligned)"
        assert torch.all(buf[:1] == 0) and torch.all(buf[1 + rows * cols:] == 0)


@pytest.mark.parametrize("cols", [4096, 16384, 32000, 131072])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place_persistent_many_rows(st, cols, dt):
    """In place with more rows than resident CTAs (persistent CTAs and
    clusters walk several rows; the bulk-copy ring prefetches later rows
    while earlier ones are written), AUTO path, and the causal variant."""
    rows = 700
    x = _inputs(rows, cols, dt, seed=cols + 31)
    ref = st.softmax(x)
    z = x.clone()
    st.softmax(z, out=z)
    torch.cuda.synchronize()
    assert torch.equal(z, ref)
    ref_c = st.softmax_causal(x, period=333, offset=5)
    z = x.clone()
    st.softmax_causal(z, period=333, offset=5, out=z)
    torch.cuda.synchronize()
    assert torch.equal(z, ref_c)


SOFTMAX_WORKLOADS = [n for n, w in workloads.WORKLOADS.items() if w.op == "softmax"]


@pytest.mark.parametrize("name", SOFTMAX_WORKLOADS)
@pytest.mark.parametrize("path", PATHS)
def test_workload_recipe_scaled(st, name, path):
    w = workloads.WORKLOADS[name]
    rows = min(w.rows, 300 if w.cols <= 4096 else 24)
    x = workloads.make(w.scaled(rows=rows), device="cuda")
    _check(st, x, w.dtype, path, f"{name} x{rows} rows, {path}")


@pytest.mark.parametrize("name", SOFTMAX_WORKLOADS)
def test_workload_full_size_all_rows(st, name):
    """Full-size input, the launch the benchmark times: every row against the
    oracle (in blocks of rows, to bound host memory), row sums and ranges, and
    a bit-identical second run."""
    w = workloads.WORKLOADS[name]
    x = workloads.make(w, device="cuda")
    y = st.softmax(x)
    torch.cuda.synchronize()
    block = max(1, (1 << 26) // w.cols)  # ~64M elements, 512 MB of float64, per block
    for r0 in range(0, w.rows, block):
        r1 = min(w.rows, r0 + block)
        xs = x[r0:r1].double().cpu().numpy()
        ys = y[r0:r1].double().cpu().numpy()
        assert_softmax_close(xs, ys, oracle.softmax(xs), w.dtype, f"{name} rows {r0}..{r1 - 1}")
    sums = y.double().sum(dim=1)
    assert float((sums - 1).abs().max()) <= SUM_TOL[w.dtype]
    assert float(y.min()) >= 0.0 and float(y.max()) <= 1.0
    assert int(torch.isnan(y).sum()) == 0
    if name.startswith("causal"):  # rows r with r % 128 == 0 have one finite entry
        assert torch.all(y[::128, 0] == 1.0) and torch.all(y[::128, 1:] == 0)
    y2 = st.softmax(x)
    assert torch.equal(y, y2), "two runs on the same input differ"


@pytest.mark.parametrize("name", ["softmax_8192x128256_bf16"])
def test_workload_full_size_poly_path(st, name):
    """The ex2.approx-free streaming kernel for bf16 results at full size:
    every row against the oracle, row sums, and agreement with the SFU kernel
    within both tolerances."""
    w = workloads.WORKLOADS[name]
    x = workloads.make(w, device="cuda")
    y = st.softmax(x, path="stream_poly")
    torch.cuda.synchronize()
    block = max(1, (1 << 26) // w.cols)
    for r0 in range(0, w.rows, block):
        r1 = min(w.rows, r0 + block)
        xs = x[r0:r1].double().cpu().numpy()
        assert_softmax_close(xs, y[r0:r1].double().cpu().numpy(), oracle.softmax(xs), w.dtype,
                             f"{name} poly rows {r0}..{r1 - 1}")
    sums = y.double().sum(dim=1)
    assert float((sums - 1).abs().max()) <= SUM_TOL[w.dtype]


@pytest.mark.parametrize("path", ["stream", "stream_poly", "safe"])
@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
def test_large_magnitude_rows(st, pair, path):
    """Rows whose maximum lies far from 0 (|m| from 1000 to 1e6, both signs):
    the bf16 kernels bound their inputs on packed pairs only while |m| < 2048
    and take the fp32 bound beyond; the folded shift must carry m log2 e
    exactly enough either way.  Spread of 60 below the maximum, a few -inf."""
    rows, cols = 10, 40000
    rng = np.random.default_rng(23)
    x64 = -rng.uniform(0.0, 60.0, size=(rows, cols))
    x64[:, 777] = 0.0
    x64[:, 100:110] = -np.inf
    x64 += np.array([1000.0, -1000.0, 2040.0, 2100.0, -2100.0, 5000.0, 3e4, -3e4, 1e6, -1e6])[:, None]
    x = torch.tensor(x64, dtype=torch.float64).to(DT[pair[0]]).cuda()
    _check(st, x, pair[1], path, f"large magnitudes {pair} {path}")


def test_edge_rows(st):
    n = 4099
    rows = []
    for pos in (0, 1, 2047, n - 1):
        r = np.full(n, -np.inf)
        r[pos] = 3.0
        rows.append(r)                              # all but one -inf
    r = np.linspace(-5, 5, n)
    r[:100] = -np.inf
    rows.append(r)                                  # -inf first, then increasing
    r = np.random.default_rng(1).normal(size=n) * 3
    r[[3, 900, 2000, 4098]] = 40.0
    rows.append(r)                                  # four exact spikes
    rows.append(np.full(n, -7.25))                  # constant
    r = np.random.default_rng(2).normal(size=n)
    r[10] = 1e30
    r[11] = -1e30
    rows.append(r)                                  # huge magnitudes
    rows.append(np.arange(n, dtype=np.float64) * 1e-3)  # strictly increasing
    x64 = np.stack(rows)
    for dtype in ("f32", "bf16"):
        x = torch.tensor(x64).to(DT[dtype]).cuda()
        for path in PATHS:
            try:
                y = st.softmax(x, path=path)
            except st.OsError as e:
                assert e.name == "OS_ERR_PATH"
                continue
            torch.cuda.synchronize()
            xx = x.double().cpu().numpy()
            assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), dtype,
                                 f"edge rows {dtype} {path}")


def test_single_column_and_spike_ties(st):
    x = torch.randn(1000, 1, device="cuda")
    assert torch.all(st.softmax(x) == 1.0)
    w = workloads.WORKLOADS["softmax_8192x128256_bf16"].scaled(rows=8)
    x = workloads.make(w, device="cuda")
    y = st.softmax(x).float()
    spikes = x.float() == 40.0
    per_row = y.masked_fill(~spikes, 0)
    for r in range(8):
        vals = per_row[r][spikes[r]]
        assert vals.numel() == 4 and torch.all(vals == vals[0]), vals


def test_all_neg_inf_row_does_not_disturb_others(st):
    x = torch.randn(6, 3000, device="cuda")
    x[2] = -np.inf
    y = st.softmax(x)
    torch.cuda.synchronize()
    keep = [0, 1, 3, 4, 5]
    xx = x[keep].double().cpu().numpy()
    assert_softmax_close(xx, y[keep].double().cpu().numpy(), oracle.softmax(xx), "f32", "others")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
def test_wide_exponent_range(st, pair, path):
    """One entry at the row maximum and the rest spread over [max - 87.3, max - 20],
    so that d stays close to 1 and e^(x - m) / d sweeps the normal fp32 range
    down to FLT_MIN: the exponential's error grows with |x - m|, and this is
    where it is largest.  Row offsets from -300 to +300 make x - m a rounded
    difference for fp32 inputs."""
    rows, cols = 12, 20000
    rng = np.random.default_rng(17)
    x64 = rng.uniform(-87.3, -20.0, size=(rows, cols))
    x64[:, 4321] = 0.0
    x64 += np.linspace(-300.0, 300.0, rows)[:, None]
    x = torch.tensor(x64, dtype=torch.float64).to(DT[pair[0]]).cuda()
    e = _check(st, x, pair[1], path, f"wide range {pair} {path}")
    assert e["max_rel"] <= {"f32": 1e-5, "bf16": 8e-3}[pair[1]]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
@pytest.mark.parametrize("cols", [100, 4096, 30000, 100000])
def test_misaligned_pointers(st, pair, cols):
    """Buffers starting 1 element past a 16-byte boundary take the element-wise path."""
    rows = 4
    xin, xout = DT[pair[0]], DT[pair[1]]
    xbuf = torch.empty(rows * cols + 8, dtype=xin, device="cuda")
    ybuf = torch.zeros(rows * cols + 8, dtype=xout, device="cuda")
    x = xbuf[1:1 + rows * cols].view(rows, cols)
    x.copy_(_inputs(rows, cols, pair[0], seed=5))
    y = ybuf[1:1 + rows * cols].view(rows, cols)
    in_code = 0 if pair[0] == "f32" else 1
    out_code = 0 if pair[1] == "f32" else 1
    st.os_softmax_fwd(x.data_ptr(), y.data_ptr(), rows, cols, in_code, out_code,
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    xx = x.double().cpu().numpy()
    assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), pair[1], "misaligned")
    assert float(ybuf[0]) == 0.0 and torch.all(ybuf[1 + rows * cols:] == 0)


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
@pytest.mark.parametrize("xoff,yoff", [(0, 0), (1, 1), (0, 3), (2, 1), (3, 0)])
@pytest.mark.parametrize("path", ["auto", "stream", "safe", "stream_poly"])
def test_rows_not_whole_vectors(st, pair, xoff, yoff, path):
    """Rows of 50257, 16387, 3001, 1001 and 257 columns (streaming, on-chip and
    warp kernels): every row starts at another offset in its 16-byte block,
    so the kernels peel the partial blocks at both ends and move the rest
    with 128-bit accesses; the output may have the input's block phase
    (vector stores) or not (element stores).  Many rows: persistent CTAs walk
    several rows and every head occurs; guard elements stay untouched."""
    for cols in (50257, 16387, 3001, 1001, 257):
        rows = 300 if cols > 20000 else (40 if cols > 10000 else 700)
        xin, xout = DT[pair[0]], DT[pair[1]]
        xbuf = torch.empty(rows * cols + 8, dtype=xin, device="cuda")
        ybuf = torch.full((rows * cols + 8,), 7.0, dtype=xout, device="cuda")
        x = xbuf[xoff:xoff + rows * cols].view(rows, cols)
        x.copy_(_inputs(rows, cols, pair[0], seed=cols + xoff))
        y = ybuf[yoff:yoff + rows * cols].view(rows, cols)
        in_code = 0 if pair[0] == "f32" else 1
        out_code = 0 if pair[1] == "f32" else 1
        try:
            st.os_softmax_fwd_path(x.data_ptr(), y.data_ptr(), rows, cols, in_code, out_code,
                                   st.PATHS[path], torch.cuda.current_stream().cuda_stream)
        except st.OsError as e:
            assert e.name == "OS_ERR_PATH"
            continue
        torch.cuda.synchronize()
        xx = x.double().cpu().numpy()
        assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), pair[1],
                             f"{path} {pair} offsets {xoff}/{yoff} cols={cols}")
        assert torch.all(ybuf[:yoff] == 7.0) and torch.all(ybuf[yoff + rows * cols:] == 7.0)


SHORT_STREAM_COLS = [257, 1000, 4097, 8191, 8192, 8193, 12000, 16385, 24575, 24576, 24577,
                     32000, 49152, 49153]


@pytest.mark.parametrize("path", ["auto", "stream", "stream_poly"])
@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
def test_stream_short_row_ctas(st, pair, path):
    """At least as many rows as SMs, rows of up to 96 KB: the streaming kernel
    runs CTAs of 256 threads (four per SM, 48 KB kept on chip), 512 beyond.
    Columns cross its chunk sizes, the kept part, the 96 KB switch (24576
    fp32, 49152 bf16) and the vector width; aligned and unaligned bases."""
    rows = 160
    esz = 4 if pair[0] == "f32" else 2
    code = (0 if pair[0] == "f32" else 1, 0 if pair[1] == "f32" else 1)
    for cols in SHORT_STREAM_COLS:
        p = st.plan((rows, cols), code[0], code[1], path=path)
        if p["path"] in (st.OS_PATH_STREAM, st.OS_PATH_STREAM_POLY):
            assert p["cluster"] == 1 and p["threads"] == (256 if cols * esz <= 96 * 1024 else 512), (cols, p)
        for off in (0, 1):
            xbuf = torch.empty(rows * cols + 8, dtype=DT[pair[0]], device="cuda")
            x = xbuf[off:off + rows * cols].view(rows, cols)
            x.copy_(_inputs(rows, cols, pair[0], seed=cols + 3 * off))
            y = torch.empty(rows, cols, dtype=DT[pair[1]], device="cuda")
            st.os_softmax_fwd_path(x.data_ptr(), y.data_ptr(), rows, cols, code[0], code[1],
                                   st.PATHS[path], torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            xx = x.double().cpu().numpy()
            assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), pair[1],
                                 f"{path} {pair} cols={cols} offset {off}")


@pytest.mark.parametrize("cols", [128, 1024, 4096, 32000, 128256, 300000])
def test_output_guard_bands_untouched(st, cols):
    rows = 7
    guard = 4096
    x = _inputs(rows, cols, "f32", seed=9)
    buf = torch.full((2 * guard + rows * cols,), 12345.0, device="cuda")
    y = buf[guard:guard + rows * cols].view(rows, cols)
    st.softmax(x, out=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 12345.0) and torch.all(buf[guard + rows * cols:] == 12345.0)
    xx = x.double().cpu().numpy()
    assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), "f32", "guarded")


def test_side_stream(st):
    s = torch.cuda.Stream()
    x = _inputs(64, 32000, "f32", seed=3)
    with torch.cuda.stream(s):
        y = st.softmax(x)
    s.synchronize()
    xx = x.double().cpu().numpy()
    assert_softmax_close(xx, y.double().cpu().numpy(), oracle.softmax(xx), "f32", "side stream")


def test_plans_of_the_workloads(st):
    p = st.plan((4096, 32000), st.OS_F32)
    assert p["path"] == st.OS_PATH_STREAM and p["cluster"] == 1
    p = st.plan((8192, 128256), st.OS_BF16)
    assert p["path"] == st.OS_PATH_STREAM and p["cluster"] == 1
    p = st.plan((8192, 128256), st.OS_BF16, path="onchip")
    assert p["path"] == st.OS_PATH_ONCHIP and p["cluster"] == 8 and p["stages"] == 3
    p = st.plan((1048576, 128), st.OS_F32)
    assert p["path"] == st.OS_PATH_WARP and p["lanes_per_row"] == 4 and p["vectors_per_thread"] == 8
    p = st.plan((65536, 4096), st.OS_F32)
    assert p["path"] == st.OS_PATH_ONCHIP and p["cluster"] == 1 and p["threads"] == 128
    # AUTO's family boundaries and the streaming kernel's CTA size
    assert st.plan((4096, 8192), st.OS_F32)["path"] == st.OS_PATH_ONCHIP
    assert st.plan((4096, 8193), st.OS_F32)["path"] == st.OS_PATH_STREAM
    assert st.plan((4096, 8192), st.OS_BF16)["path"] == st.OS_PATH_ONCHIP
    assert st.plan((4096, 8193), st.OS_BF16)["path"] == st.OS_PATH_STREAM
    assert st.plan((4096, 1024), st.OS_BF16)["path"] == st.OS_PATH_WARP
    assert st.plan((4096, 1025), st.OS_BF16)["path"] == st.OS_PATH_ONCHIP
    assert st.plan((4096, 1024), st.OS_F32)["path"] == st.OS_PATH_WARP
    assert st.plan((4096, 24576), st.OS_F32)["threads"] == 256
    assert st.plan((4096, 24577), st.OS_F32)["threads"] == 512
    assert st.plan((4096, 49152), st.OS_BF16)["threads"] == 256
    assert st.plan((100, 24576), st.OS_F32)["threads"] == 512  # fewer rows than SMs: clusters
    with pytest.raises(st.OsError):
        st.plan((10, 5000), st.OS_F32, path="warp")


def test_bad_calls_raise(st):
    x = torch.randn(4, 100, device="cuda")
    with pytest.raises(st.OsError) as e:
        st.os_softmax_fwd(x.data_ptr(), x.data_ptr() + 4, 4, 100, 0, 0, None)
    assert e.value.name == "OS_ERR_ALIAS"
    with pytest.raises(st.OsError) as e:
        st.softmax(torch.randn(2, 5000, device="cuda"), path="warp")
    assert e.value.name == "OS_ERR_PATH"
