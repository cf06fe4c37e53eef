"""Attention forward on the tensor cores against the float64 oracle.

Tolerance, from the arithmetic of the kernel.  The scores s = q . k are
fp32 sums of D exact bf16 products: |s~ - s| <= D 2^-23 sum_c |q_c k_c|
(a generous bound for the tensor core's fp32 accumulation), which moves a
probability by the factor e^(scale |s~ - s|).  Each probability p_j is taken
in fp32 (ex2 approximation, ~2^-22) and rounded to bf16 for the P V product
(relative error <= 2^-9), while l sums the fp32 values (n 2^-24 relative at
most).  So each weight w_j = p_j / l carries a relative error delta <=
2^-9 + scale D 2^-23 max_j sum_c |q_c k_jc| + n 2^-24 (computed per query
row), and
  |O~_c - O_c| <= 2 delta sum_j w_j |v_jc| + 2^-8 |O_c|,
the second term covering the final rounding of O to bf16 (2^-9).  The factor
sum_j w_j |v_jc| is the oracle's own attention output for |V|.  L = m + ln l
only sees the fp32 errors: |L~ - L| <= scale D 2^-23 max_j sum_c |q_c k_jc|
+ n 2^-23 + 2^-20 |L| + 2^-20.

Cases span several 128-row tiles with ragged tails, both head dimensions,
with and without the causal mask, scores spread wide enough that the running
maximum jumps many times (the tensor-memory rescale), and the full-size
workload checked on sampled rows plus a property of every row.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _rand(bh, n, d, seed, scale_q=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = (torch.randn(bh, n, d, generator=g, device="cuda") * scale_q).to(torch.bfloat16)
    k = torch.randn(bh, n, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(bh, n, d, generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v


def _np(t):
    return t.detach().double().cpu().numpy()


def _score_bound(q_rows, k_slices, slices, rows, scale, causal):
    """scale D 2^-23 max_j sum_c |q_c k_jc| over the keys each query row sees,
    and the number of keys it sees."""
    d = q_rows.shape[-1]
    n = k_slices.shape[1]
    out, seen = np.empty(len(rows)), np.empty(len(rows))
    for p, (b, i) in enumerate(zip(slices, rows)):
        cnt = i + 1 if causal else n
        out[p] = (np.abs(k_slices[b, :cnt]) @ np.abs(q_rows[p])).max()
        seen[p] = cnt
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return s * d * 2.0 ** -23 * out, seen


def _check(o, lse, ro, rl, abs_w, sbound, seen, label):
    o, lse = _np(o), _np(lse)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{label}: non-finite output"
    # sbound, seen: one value per query row (the shape of lse)
    delta = (2.0 ** -9 + sbound + seen * 2.0 ** -24)[..., None]
    tol = 2 * delta * abs_w + 2.0 ** -8 * np.abs(ro) + 1e-6
    err = np.abs(o - ro)
    bad = err > tol
    assert not bad.any(), (f"{label}: {bad.sum()} of {bad.size} O entries out of tolerance; "
                           f"worst err {err.max():.3e}, worst err/tol {(err / tol).max():.3f}")
    ltol = sbound + seen * 2.0 ** -23 + 2.0 ** -20 * (1 + np.abs(rl))
    lerr = np.abs(lse - rl)
    assert np.all(lerr <= ltol), (f"{label}: L worst err {lerr.max():.3e}, "
                                  f"worst err/tol {(lerr / ltol).max():.3f}")


def _full_check(st, q, k, v, causal, scale=None, label=""):
    o, lse = st.attention(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    q64, k64, v64 = _np(q), _np(k), _np(v)
    ro, rl = oracle.attention(q64, k64, v64, scale, causal)
    aw, _ = oracle.attention(q64, k64, np.abs(v64), scale, causal)
    bh, n, _ = q64.shape
    sl, rw = np.repeat(np.arange(bh), n), np.tile(np.arange(n), bh)
    sb, seen = _score_bound(q64.reshape(bh * n, -1), k64, sl, rw, scale, causal)
    _check(o, lse, ro, rl, aw, sb.reshape(bh, n), seen.reshape(bh, n), label)
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 7, 128, 130, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_matches_oracle(st, d, n, causal):
    q, k, v = _rand(3, n, d, seed=1000 + n + d + int(causal))
    _full_check(st, q, k, v, causal, label=f"n={n} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_small_workload(st, causal):
    w = workloads.ATTENTION_WORKLOADS["attention_1x2x300x64_bf16"]
    q, k, v = workloads.make_attention(w, device="cuda")
    _full_check(st, q, k, v, causal, label=f"{w.name} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_rescale_path_wide_scores(st, causal, d):
    """Queries scaled by 12: scores spread over hundreds of units in the base-2
    exponent, so many tiles raise the maximum by more than 2^8."""
    q, k, v = _rand(2, 700, d, seed=77 + d, scale_q=12.0)
    _full_check(st, q, k, v, causal, label=f"wide d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_rescale_every_tile_increasing_scores(st, causal):
    """Keys along one direction with growing length: each query's scores grow
    along the sequence, so every key tile moves the maximum."""
    bh, n, d = 2, 1030, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    u = torch.randn(bh, 1, d, generator=g, device="cuda")
    u = u / u.norm(dim=-1, keepdim=True)
    ramp = torch.linspace(0, 400, n, device="cuda")[None, :, None]
    k = (u * ramp + 0.05 * torch.randn(bh, n, d, generator=g, device="cuda")).to(torch.bfloat16)
    q = (u.expand(bh, n, d) * 2).to(torch.bfloat16).contiguous()
    v = torch.randn(bh, n, d, generator=g, device="cuda").to(torch.bfloat16)
    _full_check(st, q, k, v, causal, label=f"increasing causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_many_items_per_cta(st, d, causal):
    """More work units than SMs (200 slices of 3 query tiles, the last ragged):
    every persistent CTA walks several items, so barrier phases and buffers
    carry over from one item to the next; every row against the oracle."""
    q, k, v = _rand(200, 259, d, seed=400 + d + int(causal))
    _full_check(st, q, k, v, causal, label=f"many items d={d} causal={causal}")


def test_explicit_scale_and_equal_keys(st):
    """Equal keys: uniform weights, O = mean of the visible values; another
    scale value goes through unchanged."""
    bh, n, d = 2, 260, 128
    q, _, v = _rand(bh, n, d, seed=9)
    k = torch.ones(bh, n, d, device="cuda", dtype=torch.bfloat16) * 0.5
    for causal in (False, True):
        _full_check(st, q, k, v, causal, scale=0.3, label=f"equal keys causal={causal}")


def test_no_lse_and_repeatable(st):
    q, k, v = _rand(4, 384, 128, seed=11)
    o1, l1 = st.attention(q, k, v)
    o2, l2 = st.attention(q, k, v, want_lse=False)
    o3, _ = st.attention(q, k, v)
    torch.cuda.synchronize()
    assert l2 is None
    assert torch.equal(o1, o2) and torch.equal(o1, o3)


def test_four_dim_tensors(st):
    q, k, v = _rand(6, 200, 64, seed=12)
    o, lse = st.attention(q.view(2, 3, 200, 64), k.view(2, 3, 200, 64), v.view(2, 3, 200, 64),
                          causal=True)
    o_ref, l_ref = st.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert o.shape == (2, 3, 200, 64) and lse.shape == (2, 3, 200)
    assert torch.equal(o.view(6, 200, 64), o_ref) and torch.equal(lse.view(6, 200), l_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("start", [4096, 4104])
def test_output_does_not_touch_neighbours(st, d, start):
    """Outputs written into the middle of a larger buffer leave the guard
    regions on both sides untouched (ragged n); the output starts 32-byte
    aligned (wide row stores) or only 16-byte aligned (start = 4104 bf16)."""
    bh, n = 3, 131
    q, k, v = _rand(bh, n, d, seed=13)
    big = torch.full((bh * n * d + 2 * 4096 + 8,), 7.0, device="cuda", dtype=torch.bfloat16)
    out = big[start:start + bh * n * d].view(bh, n, d)
    lbig = torch.full((bh * n + 2 * 64,), -3.0, device="cuda", dtype=torch.float32)
    lout = lbig[64:64 + bh * n].view(bh, n)
    st.attention(q, k, v, out=out, lse=lout)
    torch.cuda.synchronize()
    assert torch.all(big[:start] == 7.0) and torch.all(big[start + bh * n * d:] == 7.0)
    assert torch.all(lbig[:64] == -3.0) and torch.all(lbig[64 + bh * n:] == -3.0)
    q64, k64, v64 = _np(q), _np(k), _np(v)
    ro, rl = oracle.attention(q64, k64, v64)
    aw, _ = oracle.attention(q64, k64, np.abs(v64))
    sl, rw = np.repeat(np.arange(bh), n), np.tile(np.arange(n), bh)
    sb, seen = _score_bound(q64.reshape(bh * n, -1), k64, sl, rw, None, False)
    _check(out, lout, ro, rl, aw, sb.reshape(bh, n), seen.reshape(bh, n), "embedded output")


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_workload_sampled_rows(st, causal):
    """The benchmark's workload at full size: every row checked against the
    convex-combination bound, and 96 sampled rows (first, last, tile edges,
    random) against the oracle row by row."""
    w = workloads.ATTENTION_WORKLOADS["attention_4x16x4096x128_bf16"]
    q, k, v = workloads.make_attention(w, device="cuda")
    o, lse = st.attention(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # each O row is a convex combination of the value rows the query sees
    vmax = v.float().abs().amax(dim=1, keepdim=True)
    assert torch.all(o.float().abs() <= vmax * (1 + 2.0 ** -7) + 1e-6)
    rng = np.random.default_rng(2024 + int(causal))
    n = w.seq_len
    rows = [0, 1, 127, 128, 129, 2047, 2048, n - 129, n - 128, n - 1]
    pairs = [(int(rng.integers(w.bh)), r) for r in rows]
    pairs += [(int(rng.integers(w.bh)), int(rng.integers(n))) for _ in range(96 - len(pairs))]
    sl = np.array([p[0] for p in pairs])
    rw = np.array([p[1] for p in pairs])
    k64, v64 = _np(k), _np(v)
    qsel = _np(q)[sl, rw]
    ro, rl = oracle.attention_rows(qsel, k64, v64, sl, rw, None, causal)
    aw, _ = oracle.attention_rows(qsel, k64, np.abs(v64), sl, rw, None, causal)
    o_sel = o[torch.as_tensor(sl, device="cuda"), torch.as_tensor(rw, device="cuda")]
    l_sel = lse[torch.as_tensor(sl, device="cuda"), torch.as_tensor(rw, device="cuda")]
    sb, seen = _score_bound(qsel, k64, sl, rw, None, causal)
    _check(o_sel, l_sel, ro, rl, aw, sb, seen, f"{w.name} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_long_ragged_sequence_sampled_rows(st, causal):
    """A long ragged sequence (n = 16389, 129 query tiles, the last holding 5
    rows): 64 sampled rows, including both ends and tile edges, against the
    oracle row by row."""
    bh, n, d = 2, 16389, 128
    q, k, v = _rand(bh, n, d, seed=900 + int(causal))
    o, lse = st.attention(q, k, v, causal=causal)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31 + int(causal))
    rows = [0, 127, 128, 8191, 16383, 16384, n - 1]
    pairs = [(r % bh, r) for r in rows] + [(int(rng.integers(bh)), int(rng.integers(n)))
                                           for _ in range(64 - len(rows))]
    sl = np.array([p[0] for p in pairs])
    rw = np.array([p[1] for p in pairs])
    k64, v64 = _np(k), _np(v)
    qsel = _np(q)[sl, rw]
    ro, rl = oracle.attention_rows(qsel, k64, v64, sl, rw, None, causal)
    aw, _ = oracle.attention_rows(qsel, k64, np.abs(v64), sl, rw, None, causal)
    sb, seen = _score_bound(qsel, k64, sl, rw, None, causal)
    idx = (torch.as_tensor(sl, device="cuda"), torch.as_tensor(rw, device="cuda"))
    _check(o[idx], lse[idx], ro, rl, aw, sb, seen, f"long n={n} causal={causal}")


def test_lse_matches_stats_kernel_on_scores(st):
    """L of a short sequence equals the row log-sum-exp of the scaled score
    matrix computed by the library's own statistics kernel from the same
    scores (a second, independent path through the library)."""
    bh, n, d = 1, 256, 64
    q, k, v = _rand(bh, n, d, seed=21)
    _, lse = st.attention(q, k, v)
    scores = (q[0].double() @ k[0].double().T / math.sqrt(d)).float().contiguous()
    _, _, lse_rows = st.softmax_stats(scores)
    torch.cuda.synchronize()
    assert torch.allclose(lse[0].double(), lse_rows.double(), atol=2.0 ** -8, rtol=0)
