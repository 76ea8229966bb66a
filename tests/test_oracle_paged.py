"""Pins of the oracle's paged read (gather_paged): a cache laid out in shuffled
pages by the input generator's scatter (synth.paginate) reads back, through
the page table, as the contiguous cache it came from; with one page per
sequence and the identity table the pool is the cache itself."""
import numpy as np
import pytest

import oracle as O
import synth


@pytest.mark.parametrize("shape,page_rows,dtype", [((3, 200, 16), 64, np.uint16),
                                                    ((2, 128, 4), 128, np.uint8),
                                                    ((4, 70, 8), 64, np.float32)])
def test_paged_cache_reads_back_as_its_contiguous_gather(shape, page_rows, dtype):
    rng = np.random.default_rng(7)
    arr = rng.integers(0, 1 << 14, size=shape).astype(dtype)
    pool, table = synth.paginate(arr, page_rows, seed=3, spare_pages=5)
    B, cap = shape[0], shape[1]
    assert table.shape == (B, -(-cap // page_rows))
    assert len(np.unique(table)) == table.size          # no page serves two places
    assert pool.shape[0] == (table.size + 5) * page_rows
    for b in range(B):
        got = O.gather_paged(pool, table[b], page_rows, cap)
        assert np.array_equal(got, arr[b])
        # and row by row from the definition
        for r in (0, cap // 2, cap - 1):
            assert np.array_equal(pool[int(table[b, r // page_rows]) * page_rows + r % page_rows],
                                  arr[b, r])


def test_identity_table_is_the_contiguous_layout():
    arr = np.arange(2 * 128 * 3, dtype=np.int32).reshape(2, 128, 3)
    pool = arr.reshape(256, 3)
    table = np.array([[0], [1]], np.int32)
    for b in range(2):
        assert np.array_equal(O.gather_paged(pool, table[b], 128, 128), arr[b])


def test_a_different_table_reads_different_rows():
    """A plausible mistake (using the logical page as the physical one) fails."""
    arr = np.arange(2 * 192, dtype=np.int64).reshape(2, 192)
    pool, table = synth.paginate(arr, 64, seed=11, spare_pages=0)
    assert not np.array_equal(table.reshape(-1), np.arange(table.size))
    wrong = np.arange(table.size).reshape(table.shape)
    assert any(not np.array_equal(O.gather_paged(pool, wrong[b], 64, 192), arr[b])
               for b in range(2))
