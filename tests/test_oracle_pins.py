"""Pins of the float64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function checks one such fact against an oracle library handle
and raises AssertionError when it does not hold.  The tests below run every pin
on the real oracle; tests/test_oracle_mutants.py runs the same pins on
deliberately broken copies of the oracle and requires each copy to fail one.

Sources of the facts (pages named by title and section):
  * Lesson 7 "Online Softmax and associative state", worked two-shard example
    and the NumPy chunked-simulation check (tests/golden/).
  * The same page, section 3: identity element (-inf, 0).
  * "Online normalizer calculation for softmax" notes, section 3.2: the
    recurrence's d equals sum_j e^(x_j - m) (induction proof) and
    1 <= d_j <= j; section 3.3: the operator is associative and commutative;
    section 4: top-K of y equals top-K of the logits (softmax is monotone).
  * "CUDA operator optimization (3): Softmax", subtract-max trick: softmax is
    invariant under adding a constant to every entry.
  * Closed forms: one entry -> 1; constant row -> 1/n; two entries -> the
    logistic function of their difference; y_i = 1 / sum_j e^(x_j - x_i).
  * "6.2 FlashAttention V2", section 6.1: the tiled forward loop (running max,
    running sum, rescaled output, final division, L = m + ln l) reaches the
    attention oracle's O and L; attention closed forms and invariants.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from tests import _golden

pytestmark = pytest.mark.filterwarnings("ignore")


def _lib():
    return oracle.load()


# ---------------------------------------------------------------- (m, d) state
def pin_two_shard_example(lib):
    g = _golden.load("two_shard_example.txt")
    step = 10.0 ** -int(g["printed_decimals"])

    def shown(value, printed):  # the page truncates after the last printed decimal
        return 0.0 <= value - printed < step

    ma, da = (v[0] for v in oracle.row_stats(g["shard_a"], lib))
    mb, db = (v[0] for v in oracle.row_stats([g["shard_b"]], lib))
    assert ma == g["m_a"] and shown(da, g["d_a"]), (ma, da)
    assert mb == g["m_b"] and shown(db, g["d_b"]), (mb, db)
    m, d = oracle.combine((ma, da), (mb, db), lib)
    assert m == g["m_ab"] and shown(d, g["d_ab"]), (m, d)
    mw, dw = (v[0] for v in oracle.row_stats(g["shard_a"] + [g["shard_b"]], lib))
    assert mw == g["m_ab"] and shown(dw, g["d_three_pass"]), (mw, dw)
    e2 = oracle.row_stats([[1.0, 3.0]], lib)[1][0] - 1.0    # e^(1-3)
    e1 = oracle.row_stats([[2.0, 3.0]], lib)[1][0] - 1.0    # e^(2-3)
    assert shown(e2, g["exp_minus_2"]) and shown(e1, g["exp_minus_1"]), (e2, e1)
    # the merged state is the whole-row state, not just close to the printed value
    assert abs(d - dw) <= 1e-15 * dw
    assert abs(dw - (math.exp(-2) + math.exp(-1) + 1.0)) <= 1e-15


def pin_identity_element(lib):
    rng = np.random.default_rng(11)
    for _ in range(50):
        s = (float(rng.normal() * 30), float(rng.uniform(1, 1e4)))
        assert oracle.combine(s, (-math.inf, 0.0), lib) == s
        assert oracle.combine((-math.inf, 0.0), s, lib) == s
    assert oracle.combine((-math.inf, 0.0), (-math.inf, 0.0), lib) == (-math.inf, 0.0)


def pin_combine_associative_commutative(lib):
    rng = np.random.default_rng(12)
    for _ in range(40):
        n = int(rng.integers(3, 40))
        x = rng.normal(size=n) * rng.choice([1.0, 10.0, 60.0])
        whole = tuple(v[0] for v in oracle.row_stats(x, lib))
        a, b = sorted(rng.choice(np.arange(1, n), 2, replace=False))
        parts = [tuple(v[0] for v in oracle.row_stats(p, lib)) for p in (x[:a], x[a:b], x[b:])]
        left = oracle.combine(oracle.combine(parts[0], parts[1], lib), parts[2], lib)
        right = oracle.combine(parts[0], oracle.combine(parts[1], parts[2], lib), lib)
        swapped = oracle.combine(parts[2], oracle.combine(parts[1], parts[0], lib), lib)
        for s in (left, right, swapped):
            assert s[0] == whole[0]
            assert abs(s[1] - whole[1]) <= 1e-12 * whole[1], (s, whole)


def pin_online_recurrence_equals_definition(lib):
    rng = np.random.default_rng(13)
    rows = [rng.normal(size=n) * s for n in (1, 2, 7, 64, 1000) for s in (1.0, 25.0)]
    rows.append(np.arange(200, dtype=float))           # new maximum at every step
    rows.append(np.arange(200, dtype=float)[::-1])     # maximum first
    rows.append(np.array([-np.inf, -np.inf, 3.0, -np.inf, 1.0]))  # leading -inf
    for x in rows:
        m, d = oracle.online_stats(x, lib)
        md, dd = (v[0] for v in oracle.row_stats(x, lib))
        assert m == md and abs(d - dd) <= 1e-12 * dd, (len(x), m, d, md, dd)


def pin_normalizer_bound(lib):
    rng = np.random.default_rng(14)
    for n in (1, 5, 100, 4096):
        x = rng.normal(size=(8, n)) * 5
        x[:, ::7] = -np.inf
        x[:, 0] = rng.normal(size=8)      # keep one finite entry per row
        finite = np.isfinite(x).sum(axis=1)
        _, d = oracle.row_stats(x, lib)
        assert np.all(d >= 1.0) and np.all(d <= finite), (d, finite)


# ---------------------------------------------------------------- softmax
def pin_lesson7_numpy_check(lib):
    g = _golden.load("lesson7_numpy_check.txt")
    x = np.array(g["input_f32"], dtype=np.float32).astype(np.float64)
    y = oracle.softmax(x, lib)[0]
    # exactly rounded reference: y_i = 1 / sum_j e^(x_j - x_i), no shift by the max
    ref = np.array([1.0 / math.fsum(math.exp(xj - xi) for xj in x) for xi in x])
    assert np.allclose(y, ref, atol=g["atol"], rtol=0)
    assert abs(math.fsum(y) - 1.0) <= g["sum_atol"]
    assert np.all(np.abs(y - ref) <= 1e-15 * ref)
    # the entry below FLT_MIN stays below it; the one just above FLT_MIN does too
    assert y[5] < np.finfo(np.float32).tiny <= y[0]


def pin_closed_forms(lib):
    assert oracle.softmax([[3.25]], lib)[0, 0] == 1.0
    for n in (1, 3, 17, 1000):
        y = oracle.softmax(np.full((1, n), -2.5), lib)[0]
        assert np.all(np.abs(y - 1.0 / n) <= 1e-15 / n)
    rng = np.random.default_rng(15)
    for a, b in rng.normal(size=(50, 2)) * 10:
        y = oracle.softmax([[a, b]], lib)[0]
        assert abs(y[0] - 1.0 / (1.0 + math.exp(b - a))) <= 1e-15
        assert abs(y[1] - 1.0 / (1.0 + math.exp(a - b))) <= 1e-15


def pin_shift_invariance(lib):
    rng = np.random.default_rng(16)
    # dyadic entries and power-of-two shifts: x + c is exact, so the output must be bit-identical
    x = np.round(rng.normal(size=(6, 33)) * 64) / 64
    y = oracle.softmax(x, lib)
    for c in (1.0, -8.0, 1024.0, 2.0 ** 20):
        assert np.array_equal(oracle.softmax(x + c, lib), y)


def pin_brute_force_tiny_rows(lib):
    rng = np.random.default_rng(17)
    for n in range(1, 9):
        for _ in range(10):
            x = rng.normal(size=n) * rng.choice([0.5, 5.0, 40.0])
            if n > 2:
                x[rng.integers(n)] = -np.inf
                x[rng.integers(n)] = x.max() if np.isfinite(x.max()) else 0.0
            y = oracle.softmax(x, lib)[0]
            for i in range(n):
                if x[i] == -np.inf:
                    assert y[i] == 0.0
                    continue
                ref = 1.0 / math.fsum(math.exp(xj - x[i]) for xj in x if xj != -np.inf)
                assert abs(y[i] - ref) <= 1e-14 * ref, (x, i, y[i], ref)
            assert abs(math.fsum(y) - 1.0) <= 1e-14


def pin_rows_sum_to_one(lib):
    rng = np.random.default_rng(18)
    x = rng.normal(size=(20, 5000)) * 8
    x[rng.random(x.shape) < 0.05] = -np.inf
    x[:, 17] = 1.0
    y = oracle.softmax(x, lib)
    for row in y:
        assert abs(math.fsum(row) - 1.0) <= 1e-12


def pin_causal_and_spike_rows(lib):
    rng = np.random.default_rng(19)
    n = 128
    x = rng.normal(size=(n, n))
    x[np.arange(n)[None, :] > np.arange(n)[:, None]] = -np.inf
    y = oracle.softmax(x, lib)
    assert y[0, 0] == 1.0 and np.all(y[0, 1:] == 0.0)
    assert np.all(y[np.arange(n)[None, :] > np.arange(n)[:, None]] == 0.0)
    # four exact +40 ties: each spike is 1 / (4 + sum of the rest scaled by e^(x - 40))
    x = rng.normal(size=300) * 3
    spikes = [5, 90, 170, 299]
    x[spikes] = 40.0
    y = oracle.softmax(x, lib)[0]
    rest = math.fsum(math.exp(v - 40.0) for i, v in enumerate(x) if i not in spikes)
    for s in spikes:
        assert abs(y[s] - 1.0 / (4.0 + rest)) <= 1e-15
    assert len(set(y[spikes])) == 1


# ---------------------------------------------------------------- TopK
def _exhaustive_topk(x, K):
    """Pick the best remaining entry K times: larger logit, then lower index."""
    taken, out = set(), []
    for _ in range(K):
        best = None
        for j, v in enumerate(x):
            if j in taken:
                continue
            if best is None or v > x[best]:
                best = j
        taken.add(best)
        out.append(best)
    return out


def pin_topk_exhaustive(lib):
    rng = np.random.default_rng(20)
    for n in (1, 2, 5, 9, 33, 70):
        for _ in range(6):
            x = np.round(rng.normal(size=n) * 3, 1)        # coarse values: many ties
            if n > 3:
                x[rng.integers(n, size=2)] = -np.inf
            for K in sorted({1, min(n, 3), min(n, 8), n}):
                vals, idx = oracle.topk(x, K, lib)
                assert list(idx[0]) == _exhaustive_topk(list(x), K), (x, K, idx)
                y = oracle.softmax(x, lib)[0]
                assert np.array_equal(vals[0], y[idx[0]])


def pin_topk_ties_lower_index(lib):
    x = np.array([[0.5, 2.0, 2.0, -1.0, 2.0, 2.0, 0.5, -np.inf, -np.inf]])
    vals, idx = oracle.topk(x, 9, lib)
    assert list(idx[0]) == [1, 2, 4, 5, 0, 6, 3, 7, 8]
    assert vals[0, 0] == vals[0, 3] and vals[0, 7] == 0.0 and vals[0, 8] == 0.0


# ---------------------------------------------------------------- log-sum-exp
def pin_lse_fsum_and_closed_forms(lib):
    """lse = ln sum e^x: against an exactly rounded sum on small rows, the
    constant-row closed form c + ln n, a dyadic shift, and m <= lse <= m + ln n."""
    rng = np.random.default_rng(21)
    for n in (1, 2, 3, 7, 40):
        for _ in range(8):
            x = rng.normal(size=n) * rng.choice([0.5, 4.0, 30.0])
            got = oracle.lse(x, lib)[0]
            ref = math.log(math.fsum(math.exp(v) for v in x))
            assert abs(got - ref) <= 1e-13 * max(1.0, abs(ref)), (x, got, ref)
            assert x.max() <= got <= x.max() + math.log(n) + 1e-14
            assert abs(oracle.lse(x + 8.0, lib)[0] - (got + 8.0)) <= 1e-13 * max(1.0, abs(got))
    for c, n in ((0.0, 1), (-3.25, 10), (100.0, 4096)):
        assert abs(oracle.lse(np.full(n, c), lib)[0] - (c + math.log(n))) <= 1e-13 * max(1, abs(c))
    x = np.array([[1.0, -np.inf, 2.0], [-np.inf, -np.inf, -np.inf]])
    got = oracle.lse(x, lib)
    assert abs(got[0] - math.log(math.e + math.e ** 2)) <= 1e-15 and got[1] == -np.inf


# ---------------------------------------------------------------- causal mask
def pin_causal_mask_rows(lib):
    """Row r keeps columns c <= (r mod period) + offset: masked entries are
    exactly 0, the kept prefix is the brute-force softmax of that prefix, and a
    row that keeps only column 0 is [1, 0, ...]."""
    rng = np.random.default_rng(22)
    for period, offset, cols in ((4, 0, 4), (6, 2, 9), (3, 0, 8), (5, 10, 7)):
        x = rng.normal(size=(2 * period + 1, cols)) * 3
        masked = oracle.causal_mask(x, period, offset, lib)
        y = oracle.softmax_causal(x, period, offset, lib)
        for r in range(x.shape[0]):
            lim = min(cols, r % period + offset + 1)
            assert np.all(masked[r, lim:] == -np.inf) and np.array_equal(masked[r, :lim], x[r, :lim])
            assert np.all(y[r, lim:] == 0.0)
            for i in range(lim):
                ref = 1.0 / math.fsum(math.exp(x[r, j] - x[r, i]) for j in range(lim))
                assert abs(y[r, i] - ref) <= 1e-14 * ref
            if lim == 1:
                assert y[r, 0] == 1.0


# ---------------------------------------------------------------- top-K sampling
def pin_topk_sample_frequencies(lib):
    """With u on a grid of N midpoints the draws split in proportion to the
    values (exactly: no cumulative sum lies near a grid point); zero-probability
    entries are never drawn,
    also at u = 0; scaling all values changes nothing; u = 1 gives the last."""
    N = 1024
    u = (np.arange(N) + 0.5) / N
    for p, want in (([0.5, 0.25, 0.125, 0.125], [512, 256, 128, 128]),
                    ([1.0, 0.5, 0.25, 0.25], [512, 256, 128, 128]),
                    ([0.5, 0.0, 0.5], [512, 0, 512]),
                    ([0.75, 0.25], [768, 256]),
                    # not dyadic: the cumulative sums 0.1, 0.3, 0.6 fall between grid
                    # points (102.4, 307.2, 614.4 of 1024), far from any rounding
                    ([0.1, 0.2, 0.3, 0.4], [102, 205, 307, 410])):
        K = len(p)
        vals = np.tile(np.array(p), (N, 1))
        idx = np.tile(np.arange(K, dtype=np.int32) + 10, (N, 1))
        got = oracle.topk_sample(vals, idx, u, lib)
        assert list(np.bincount(got - 10, minlength=K)) == want, (p, np.bincount(got - 10))
    vals = np.array([[0.0, 0.3, 0.7], [0.0, 0.3, 0.7], [0.2, 0.3, 0.5]])
    idx = np.array([[5, 6, 7]] * 3, dtype=np.int32)
    assert list(oracle.topk_sample(vals, idx, [0.0, 1.0, 0.2], lib)) == [6, 7, 6]


# ---------------------------------------------------------------- attention
def _tiled_attention(q, k, v, scale, causal, Br, Bc):
    """The forward loop of "6.2 FlashAttention V2" (section 6.1) in plain
    Python: query tiles of Br rows, key/value tiles of Bc rows, running row
    maximum m, running sum l and unnormalised output, the masked key range
    ending at the query tile's end, and O = O~ / l, L = m + ln l at the end."""
    n, dh = len(q), len(q[0])
    O = [[0.0] * dh for _ in range(n)]
    L = [0.0] * n
    for i0 in range(0, n, Br):
        rows = range(i0, min(n, i0 + Br))
        m = {r: -math.inf for r in rows}
        l = {r: 0.0 for r in rows}
        acc = {r: [0.0] * dh for r in rows}
        kv_end = min(n, i0 + Br) if causal else n
        for j0 in range(0, kv_end, Bc):
            cols = range(j0, min(kv_end, j0 + Bc))
            for r in rows:
                s = [scale * sum(q[r][c] * k[j][c] for c in range(dh)) for j in cols]
                s = [-math.inf if causal and j > r else sj for sj, j in zip(s, cols)]
                m_new = max([m[r]] + s)
                p = [math.exp(sj - m_new) for sj in s]
                corr = math.exp(m[r] - m_new)
                l[r] = corr * l[r] + sum(p)
                acc[r] = [corr * a + sum(pj * v[j][c] for pj, j in zip(p, cols))
                          for c, a in enumerate(acc[r])]
                m[r] = m_new
        for r in rows:
            O[r] = [a / l[r] for a in acc[r]]
            L[r] = m[r] + math.log(l[r])
    return O, L


def pin_attention_tiled_recurrence(lib):
    """The oracle's attention equals the FlashAttention-2 tiled forward loop,
    run in plain Python on tiny heads with ragged tiles, with and without the
    causal mask, for the default 1/sqrt(dh) scale and another one."""
    rng = np.random.default_rng(31)
    for n, dh, Br, Bc in ((7, 3, 3, 2), (5, 4, 2, 3), (1, 2, 1, 1), (9, 2, 4, 4)):
        q, k, v = (rng.normal(size=(2, n, dh)) * 2 for _ in range(3))
        for causal in (False, True):
            for scale in (None, 0.7):
                o, L = oracle.attention(q, k, v, scale, causal, lib=lib)
                sc = 1.0 / math.sqrt(dh) if scale is None else scale
                refs = []
                for b in range(2):
                    O_ref, L_ref = _tiled_attention(q[b].tolist(), k[b].tolist(), v[b].tolist(),
                                                    sc, causal, Br, Bc)
                    refs.append((np.array(O_ref), np.array(L_ref)))
                    assert np.allclose(o[b], O_ref, rtol=1e-12, atol=1e-12), (n, dh, causal)
                    assert np.allclose(L[b], L_ref, rtol=1e-12, atol=1e-12), (n, dh, causal)
                # the selected-rows entry: pairs in scrambled order
                sl = np.array([1, 0, 1, 0])
                rw = np.array([n - 1, 0, n // 2, n - 1])
                o2, L2 = oracle.attention_rows(q[sl, rw], k, v, sl, rw, scale, causal, lib=lib)
                for p, (b, i) in enumerate(zip(sl, rw)):
                    assert np.allclose(o2[p], refs[b][0][i], rtol=1e-12, atol=1e-12), (b, i)
                    assert np.allclose(L2[p], refs[b][1][i], rtol=1e-12, atol=1e-12), (b, i)


def pin_attention_closed_forms(lib):
    """One key: O = v_0 and L = scale q.k_0.  Equal keys: uniform weights over
    the keys a query sees, so O_i is the mean of those v_j (all of them, or
    j <= i under the mask) and L_i = s + ln(count).  A key that scores 200
    above the rest: O equals its value row to rounding."""
    rng = np.random.default_rng(32)
    q, k, v = (rng.normal(size=(3, 1, 5)) for _ in range(3))
    o, L = oracle.attention(q, k, v, 0.5, lib=lib)
    assert np.allclose(o, v, rtol=0, atol=1e-15)
    assert np.allclose(L[:, 0], 0.5 * np.einsum("bd,bd->b", q[:, 0], k[:, 0]), rtol=1e-14)
    n, dh = 6, 4
    q = rng.normal(size=(1, n, dh))
    k = np.tile(rng.normal(size=(1, 1, dh)), (1, n, 1))
    v = rng.normal(size=(1, n, dh))
    for causal in (False, True):
        o, L = oracle.attention(q, k, v, 1.5, causal, lib=lib)
        for i in range(n):
            cnt = i + 1 if causal else n
            s = 1.5 * float(q[0, i] @ k[0, 0])
            assert np.allclose(o[0, i], v[0, :cnt].mean(0), rtol=1e-13, atol=1e-14), (causal, i)
            assert abs(L[0, i] - (s + math.log(cnt))) <= 1e-13 * max(1.0, abs(s)), (causal, i)
    q = np.zeros((1, 4, 2))
    q[0, :, 0] = 1.0
    k = np.zeros((1, 4, 2))
    k[0, 2, 0] = 200.0  # scores 0, 0, 200, 0 for every query
    v = rng.normal(size=(1, 4, 2))
    o, _ = oracle.attention(q, k, v, 1.0, lib=lib)
    assert np.allclose(o[0], np.tile(v[0, 2], (4, 1)), rtol=0, atol=1e-15)


def pin_attention_softmax_times_v(lib):
    """O = softmax(scale Q K^T) V with the oracle's own pinned softmax applied
    to scores from a numpy matmul, and the mask applied by the pinned causal
    mask (period n); L from the pinned log-sum-exp."""
    rng = np.random.default_rng(33)
    for bh, n, dh in ((3, 17, 8), (1, 40, 16)):
        q, k, v = (rng.normal(size=(bh, n, dh)) for _ in range(3))
        for causal in (False, True):
            o, L = oracle.attention(q, k, v, None, causal, lib=lib)
            for b in range(bh):
                s = (q[b] @ k[b].T) / math.sqrt(dh)
                if causal:
                    s = oracle.causal_mask(s, n, 0, lib)
                p = oracle.softmax(s, lib)
                assert np.allclose(o[b], p @ v[b], rtol=1e-12, atol=1e-13), (b, causal)
                assert np.allclose(L[b], oracle.lse(s, lib), rtol=1e-13, atol=1e-13), (b, causal)


def pin_attention_invariants(lib):
    """Weights sum to 1, so adding c to every value row adds c to O; without the
    mask, permuting keys and values together leaves O and L alone; scaling
    values scales O; and under the mask row i depends only on keys j <= i."""
    rng = np.random.default_rng(34)
    bh, n, dh = 2, 11, 6
    q, k, v = (rng.normal(size=(bh, n, dh)) * 1.5 for _ in range(3))
    o, L = oracle.attention(q, k, v, lib=lib)
    c = rng.normal(size=dh)
    assert np.allclose(oracle.attention(q, k, v + c, lib=lib)[0], o + c, rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.attention(q, k, 3 * v, lib=lib)[0], 3 * o, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(n)
    o2, L2 = oracle.attention(q, k[:, perm], v[:, perm], lib=lib)
    assert np.allclose(o2, o, rtol=1e-12, atol=1e-12) and np.allclose(L2, L, rtol=1e-13)
    oc, Lc = oracle.attention(q, k, v, causal=True, lib=lib)
    for i in (0, 4, n - 1):
        oi, Li = oracle.attention(q[:, : i + 1], k[:, : i + 1], v[:, : i + 1], lib=lib)
        assert np.allclose(oc[:, i], oi[:, i], rtol=1e-12, atol=1e-12), i
        assert np.allclose(Lc[:, i], Li[:, i], rtol=1e-13, atol=1e-13), i
    assert np.allclose(oc[:, n - 1], o[:, n - 1], rtol=1e-12, atol=1e-12)


def pin_attention_hard_limit(lib):
    """With a huge scale the weights become one-hot on each query's best key
    (distinct scores): O is that key's value row and L the scaled best score,
    with the mask limiting the keys each query sees."""
    rng = np.random.default_rng(35)
    bh, n, dh = 2, 9, 4
    q, k, v = (rng.normal(size=(bh, n, dh)) for _ in range(3))
    scale = 1e6
    for causal in (False, True):
        o, L = oracle.attention(q, k, v, scale, causal, lib=lib)
        for b in range(bh):
            for i in range(n):
                cnt = i + 1 if causal else n
                s = k[b, :cnt] @ q[b, i]
                j = int(np.argmax(s))
                assert np.allclose(o[b, i], v[b, j], rtol=0, atol=1e-12), (b, i, causal)
                assert abs(L[b, i] - scale * s[j]) <= 1e-9 * abs(scale * s[j]) + 1e-9


PINS = [pin_two_shard_example, pin_identity_element, pin_combine_associative_commutative,
        pin_online_recurrence_equals_definition, pin_normalizer_bound, pin_lesson7_numpy_check,
        pin_closed_forms, pin_shift_invariance, pin_brute_force_tiny_rows, pin_rows_sum_to_one,
        pin_causal_and_spike_rows, pin_topk_exhaustive, pin_topk_ties_lower_index,
        pin_lse_fsum_and_closed_forms, pin_causal_mask_rows, pin_topk_sample_frequencies,
        pin_attention_tiled_recurrence, pin_attention_closed_forms, pin_attention_softmax_times_v,
        pin_attention_invariants, pin_attention_hard_limit]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(_lib())


def test_oracle_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4)), 5)
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4)), 0)


def test_oracle_threads_reported():
    assert oracle.num_threads() >= 1


def test_oracle_results_do_not_depend_on_threads():
    """Rows are independent: one thread and the default count give the same
    bits (the single-thread timing in the bench runs the same arithmetic)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((37, 1001)) * 3.0
    x[5, 100:200] = -np.inf
    cores = oracle.num_threads()
    ref_y, ref_tk = oracle.softmax(x), oracle.topk(x, 9)
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1 or cores == 1
        y, tk = oracle.softmax(x), oracle.topk(x, 9)
    finally:
        oracle.set_num_threads(cores)
    assert oracle.num_threads() == cores
    assert np.array_equal(y, ref_y)
    assert np.array_equal(tk[0], ref_tk[0]) and np.array_equal(tk[1], ref_tk[1])


def test_exhaustive_helper_itself():
    # the helper is tested on a case small enough to check by hand
    assert _exhaustive_topk([1.0, 3.0, 3.0, 2.0], 4) == [1, 2, 3, 0]
    for perm in itertools.permutations([0.0, 1.0, 2.0]):
        assert _exhaustive_topk(list(perm), 1) == [perm.index(2.0)]
