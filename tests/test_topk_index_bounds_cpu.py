"""The fused TopK kernel's index arithmetic at the longest row the C ABI
accepts (cols = 2^31 - 1), restated on the host.

A GPU run of one such row takes minutes, and a 32-bit index that wrapped there
once read far outside the row.  This test evaluates, for every cluster size
the launch plan can choose (1..8 CTAs per row), every cluster rank and every
start offset of the row inside its 16-byte block, each integer expression
that topk_rows_kernel keeps in a 32-bit int: block ranges, chunk counts, the
block indices of pass 1 and of the listing, the candidate column, and the
element loops of the exact path (which step 64-bit indices).  Every 32-bit
value must lie in int32 range, every element read must lie inside the row,
and the ranks' exact-path ranges must tile the row.
"""
import pytest

INT32_MIN, INT32_MAX = -2 ** 31, 2 ** 31 - 1
THREADS, U = 512, 4          # the kernel's CTA width and 16-byte blocks per thread per chunk
CHUNK = THREADS * U          # blocks per chunk
GROUPS = 4                   # block-key groups per thread slot
MAX_COLS = INT32_MAX


def i32(v, what):
    assert INT32_MIN <= v <= INT32_MAX, f"{what} = {v} overflows int32"
    return v


def segment(cols, head, S, rank):
    """The CTA's segment of a row, as the kernel computes it (TopkSegment)."""
    span = cols + head                               # int64
    nb = i32((span + 3) >> 2, "nb")
    full_lo = 1 if head > 0 else 0
    full_hi = i32(span >> 2, "full_hi")
    per = i32(nb + S - 1, "nb + S - 1") // S
    b0 = min(i32(rank * per, "rank * per"), nb)
    b1 = min(i32(b0 + per, "b0 + per"), nb)
    return nb, full_lo, full_hi, b0, b1


def check_pass1_and_listing(cols, head, b0, b1, full_lo, full_hi):
    nchunks = i32(b1 - b0 + CHUNK - 1, "chunk count numerator") // CHUNK
    G = max(1, (nchunks + GROUPS - 1) // GROUPS)
    i32((nchunks + G - 1), "group count numerator")
    if nchunks == 0:
        return
    # the largest and smallest block index any thread forms in pass 1 and in
    # the listing: b = b0 + c * CHUNK + k * THREADS + tid
    hi_b = i32(b0 + (nchunks - 1) * CHUNK + (U - 1) * THREADS + THREADS - 1, "pass-1 block")
    assert hi_b >= b0
    # blocks read with one 16-byte load lie wholly inside the row
    for b in (max(b0, full_lo), min(b1, full_hi) - 1):
        if full_lo <= b < full_hi and b0 <= b < b1:
            first, last = 4 * b - head, 4 * b + 3 - head
            assert 0 <= first and last <= cols - 1, (b, first, last)
    # partial blocks are read element by element, only at columns inside the row;
    # a candidate's column is formed as uint32 4b + l - head and cast to int
    for b in {b0, b1 - 1, full_lo - 1, full_hi}:
        if not (b0 <= b < b1):
            continue
        for lane in range(4):
            col = 4 * b + lane - head
            if 0 <= col < cols:
                u32 = (4 * b + lane - head) % 2 ** 32
                assert u32 <= INT32_MAX and u32 == col


def exact_path_range(cols, head, b0, b1):
    c_lo = i32(max(0, 4 * b0 - head), "c_lo")
    c_hi = i32(min(cols, 4 * b1 - head), "c_hi")
    i32(c_hi - c_lo, "c_hi - c_lo")
    if c_hi > c_lo:
        # e steps by THREADS from c_lo + tid in 64 bits: the last value formed
        # (the first past c_hi) is below c_hi + THREADS and never wraps; every
        # element read lies in [c_lo, c_hi), and int(e) of a candidate fits
        last_formed = c_hi - 1 + THREADS
        assert last_formed < 2 ** 63
        assert 0 <= c_lo and c_hi <= cols and c_hi - 1 <= INT32_MAX
    return c_lo, c_hi


@pytest.mark.parametrize("S", range(1, 9))
@pytest.mark.parametrize("head", range(4))
def test_longest_row_index_arithmetic(S, head):
    cols = MAX_COLS
    covered = []
    for rank in range(S):
        nb, full_lo, full_hi, b0, b1 = segment(cols, head, S, rank)
        check_pass1_and_listing(cols, head, b0, b1, full_lo, full_hi)
        c_lo, c_hi = exact_path_range(cols, head, b0, b1)
        if c_hi > c_lo:
            covered.append((c_lo, c_hi))
    covered.sort()
    assert covered[0][0] == 0 and covered[-1][1] == cols
    for (a0, a1), (b0, b1) in zip(covered, covered[1:]):
        assert a1 == b0, "exact-path ranges of neighbouring ranks must meet"


@pytest.mark.parametrize("cols", [1, 2, 3, 5, 4097, 50257, 2 ** 31 - 5, 2 ** 31 - 2])
@pytest.mark.parametrize("S", [1, 2, 3, 7, 8])
def test_segments_tile_the_row(cols, S):
    """Shorter and near-maximal rows: the exact-path ranges of the ranks tile
    [0, cols) for every start offset (ranks past the row's end get nothing)."""
    for head in range(4):
        ends = []
        for rank in range(S):
            _, full_lo, full_hi, b0, b1 = segment(cols, head, S, rank)
            check_pass1_and_listing(cols, head, b0, b1, full_lo, full_hi)
            c_lo, c_hi = exact_path_range(cols, head, b0, b1)
            if c_hi > c_lo:
                ends.append((c_lo, c_hi))
        assert ends[0][0] == 0 and ends[-1][1] == cols
        assert all(a[1] == b[0] for a, b in zip(ends, ends[1:]))
