"""The fp32 index arithmetic of the element-wise kernels' flat walk, checked
exhaustively on the CPU.

A tile of whole rows (W <= 1024 columns, at most 256 rows) is streamed by
flat index e, and the kernels recover the row as
    i = (int)((float(e) + 0.5f) * (1.0f / W))
with each operation rounded to nearest in fp32 (numpy's float32 operations
round the same way).  This must equal e // W for every W <= 1024 and
e < 256 W; the column is then e - i W.  The staged pass-1 chunks must fit
the 8192-value shared-memory stage and start on 4-value boundaries.
"""
import numpy as np

TILE_ROWS = 256
TILE_COLS = 1024
STAGE = 8 * 1024  # kWarps * kTileCols floats


def test_row_index_is_exact_for_every_width():
    for w in range(1, TILE_COLS + 1):
        e = np.arange(TILE_ROWS * w, dtype=np.int64)
        invw = np.float32(1.0) / np.float32(w)
        i = ((e.astype(np.float32) + np.float32(0.5)) * invw).astype(np.int64)
        assert np.array_equal(i, e // w), w


def test_staged_chunks_fit_and_stay_aligned():
    for w in range(1, TILE_COLS + 1):
        for nr in (1, 2, 3, 4, 5, 7, 8, 9, 31, 64, 100, 255, 256):
            rows_per_chunk = min(nr, (STAGE // w) & ~3)
            assert rows_per_chunk >= 1
            covered, r0 = 0, 0
            while r0 < nr:
                rows = min(rows_per_chunk, nr - r0)
                cn = rows * w
                assert cn <= STAGE
                assert cn - 4 * (cn // 4) <= 3  # the scalar tail of a chunk
                if rows_per_chunk < nr:
                    assert (r0 * w) % 4 == 0  # chunk starts on a 4-value boundary
                covered += rows
                r0 += rows_per_chunk
            assert covered == nr
