"""The streaming softmax's L2 prefetch of a CTA's next row, restated on the
host.

When a CTA's second pass over a row begins it asks L2 for the start of its
next row (`cp.async.bulk.prefetch.L2`), in pieces of 16 KB issued by its
first threads.  A bulk prefetch wants a 16-byte aligned address and a size
that is a positive multiple of 16, and nothing outside the input may be
named.  This test evaluates the kernel's address arithmetic for every CTA
size and dtype it is built for, row lengths from 1 column up to 2^31 - 1,
every base offset inside a 16-byte block, and the last rows of a launch:
every piece must be aligned, a multiple of 16 bytes, inside the next row
(so inside the input), issued only when that row exists, and the pieces of
one row must not overlap.
"""
import pytest

PIECE = 16 * 1024


def prefetch_bytes_per_thread(esz, threads):
    """The kernel's stream_prefetch_bytes_per_thread<TI, THREADS>()."""
    return 64 if esz == 2 else (192 if threads == 512 else 0)


def pieces(base, row, rows, nclusters, cols, esz, threads):
    """(address, size) of each piece the CTA issues after its row `row`,
    exactly as the kernel forms them (threads tid < NPF, a < hi)."""
    npf = threads * prefetch_bytes_per_thread(esz, threads) // PIECE
    nxt = row + nclusters
    out = []
    if npf == 0 or nxt >= rows:
        return out
    for tid in range(min(npf, threads)):
        r0 = base + nxt * cols * esz
        lo = (r0 + 15) & ~15
        hi = (r0 + cols * esz) & ~15
        a = lo + tid * PIECE
        if a < hi:
            out.append((a, min(PIECE, hi - a)))
    return out


@pytest.mark.parametrize("esz", [4, 2])
@pytest.mark.parametrize("threads", [256, 512])
@pytest.mark.parametrize("cols", [1, 3, 4, 7, 8, 1001, 8193, 24577, 32000, 50257, 128256,
                                  2 ** 20 + 3, 2 ** 31 - 1])
@pytest.mark.parametrize("offset_elems", [0, 1, 2, 3, 5, 7])
def test_pieces_aligned_inside_next_row(esz, threads, cols, offset_elems):
    base = 0x7f0000000000 + offset_elems * esz     # allocation start plus the caller's offset
    rows = 5
    nclusters = 2
    for row in range(rows):
        got = pieces(base, row, rows, nclusters, cols, esz, threads)
        nxt = row + nclusters
        if nxt >= rows:
            assert got == [], "a prefetch past the last row"
            continue
        row_lo = base + nxt * cols * esz
        row_hi = row_lo + cols * esz
        prev_end = None
        for a, size in got:
            assert a % 16 == 0 and size % 16 == 0 and size > 0, (a, size)
            assert row_lo <= a and a + size <= row_hi, "piece outside the next row"
            assert base <= a and a + size <= base + rows * cols * esz, "piece outside the input"
            assert prev_end is None or a >= prev_end, "pieces overlap"
            prev_end = a + size
        want = min(threads * prefetch_bytes_per_thread(esz, threads),
                   max(0, ((row_hi & ~15) - ((row_lo + 15) & ~15))))
        assert sum(s for _, s in got) == want


def test_no_prefetch_for_fp32_rows_on_256_thread_ctas():
    assert pieces(0, 0, 10, 1, 20000, 4, 256) == []
    assert len(pieces(0, 0, 10, 1, 20000, 2, 256)) == 1        # bf16: 16 KB
    assert len(pieces(0, 0, 10, 1, 32000, 4, 512)) == 6        # fp32: 96 KB
    assert len(pieces(0, 0, 10, 1, 128256, 2, 512)) == 2       # bf16: 32 KB
