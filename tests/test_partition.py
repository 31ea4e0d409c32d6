"""Row partitioning for data-parallel workers (spmm_partition_rows), on the host.

The partitioner is host code in the library (no CUDA call), so these run
without a GPU. The work of a row is its entry count plus one; bound q is the
first row whose prefix work reaches q/P of the total, rounded to the nearest
multiple of align_rows. The pins below are fixed by that definition and by
arithmetic, not by re-running it: even splits of uniform graphs, the
overshoot bound of a first-reach rule, whole heavy rows, alignment, and
rejection of arrays that are not row pointers.
"""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def sdm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_dense_matrix_gb300 as m
    return m


def _rowptr(degrees):
    return np.concatenate([[0], np.cumsum(degrees)]).astype(np.int32)


def test_uniform_degrees_split_evenly(sdm):
    rp = _rowptr(np.full(1000, 7))
    assert sdm.spmm_partition_rows(rp, 4) == [0, 250, 500, 750, 1000]
    assert sdm.spmm_partition_rows(rp, 1) == [0, 1000]
    # eight rows of work 8 each over three parts: targets 21.33 and 42.67 are
    # first reached after rows 3 (work 24) and 6 (work 48)
    assert sdm.spmm_partition_rows(_rowptr(np.full(8, 7)), 3) == [0, 3, 6, 8]


def test_empty_rows_still_split_by_row_count(sdm):
    rp = np.zeros(101, np.int32)              # 100 rows, no entries: work 1 per row
    assert sdm.spmm_partition_rows(rp, 4) == [0, 25, 50, 75, 100]
    assert sdm.spmm_partition_rows(np.zeros(1, np.int32), 3) == [0, 0, 0, 0]   # M = 0


def test_heavy_row_is_kept_whole_and_the_rest_balances(sdm):
    deg = np.ones(1000, np.int64)
    deg[500] = 100_000                        # one hub row holding ~98% of the work
    b = sdm.spmm_partition_rows(_rowptr(deg), 4)
    owners = [q for q in range(4) if b[q] <= 500 < b[q + 1]]
    assert len(owners) == 1                   # exactly one worker owns the hub
    # every other part gets only rows before or after it
    assert b[0] == 0 and b[-1] == 1000 and all(x <= y for x, y in zip(b, b[1:]))


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("parts", [2, 3, 7, 16])
def test_balance_and_order_on_skewed_degrees(sdm, seed, parts):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 5000))
    # a mix of empty rows, short rows and a Pareto tail
    deg = np.where(rng.random(M) < 0.3, 0, np.minimum(rng.pareto(1.2, M) * 3, 20000)).astype(np.int64)
    rp = _rowptr(deg)
    b = sdm.spmm_partition_rows(rp, parts)
    assert len(b) == parts + 1 and b[0] == 0 and b[-1] == M
    assert all(x <= y for x, y in zip(b, b[1:]))
    work = rp.astype(np.int64) + np.arange(M + 1)      # prefix work: entries + rows
    total = int(work[-1])
    w_max = int((deg + 1).max())
    # a first-reach rule overshoots its share by less than one row's work
    for q in range(parts):
        part = int(work[b[q + 1]] - work[b[q]])
        assert part < total / parts + 1 + w_max, (q, part, total / parts, w_max)
    # and every bound is the first row to reach its target
    for q in range(1, parts):
        t = q * total // parts
        assert work[b[q]] >= t and (b[q] == 0 or work[b[q] - 1] < t)


def test_alignment(sdm):
    rp = _rowptr(np.full(10_000, 10))
    b = sdm.spmm_partition_rows(rp, 3, align_rows=256)
    assert b[0] == 0 and b[-1] == 10_000
    assert all(x % 256 == 0 for x in b[1:-1]) and b[1:-1] == [3328, 6656]   # 3333, 6667 rounded
    # a granule larger than the matrix leaves the inner bounds at 0 or M
    assert sdm.spmm_partition_rows(_rowptr(np.full(100, 3)), 2, align_rows=1024) in \
        ([0, 0, 100], [0, 100, 100])


def test_rejects_what_is_not_a_row_pointer_array(sdm):
    with pytest.raises(sdm.SpmmError) as e:
        sdm.spmm_partition_rows(np.array([1, 2, 3], np.int32), 2)     # rowptr[0] != 0
    assert e.value.name == "SPMM_ERR_INVALID_INPUT"
    with pytest.raises(sdm.SpmmError) as e:
        sdm.spmm_partition_rows(np.array([0, 5, 3], np.int32), 2)     # decreasing
    assert e.value.name == "SPMM_ERR_INVALID_INPUT"
    with pytest.raises(ValueError):
        sdm.spmm_partition_rows(np.array([0, 1], np.int32), 0)
    with pytest.raises(sdm.SpmmError):
        sdm.spmm_partition_rows(np.array([0, 1], np.int32), 2, align_rows=0)
