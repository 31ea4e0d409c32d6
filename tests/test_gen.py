"""Invariants of the seeded input generators (structure the workloads promise)."""
import numpy as np
import pytest

import gen


def _check_csr(g):
    assert g.rowptr.dtype == np.int32 and g.col.dtype == np.int32
    assert g.rowptr[0] == 0 and len(g.rowptr) == g.M + 1
    assert np.all(np.diff(g.rowptr.astype(np.int64)) >= 0)
    assert g.nnz == len(g.col)
    assert g.col.min(initial=0) >= 0 and g.col.max(initial=0) < g.K
    rows = np.repeat(np.arange(g.M), g.degrees())
    # ascending and distinct within each row
    assert np.all((np.diff(g.col.astype(np.int64)) > 0) | (np.diff(rows) > 0))
    if g.val is not None:
        assert g.val.dtype == np.float32 and len(g.val) == g.nnz


def test_reproducible_and_seed_dependent():
    a, b = gen.erdos_renyi(100, 80, 5, seed=3), gen.erdos_renyi(100, 80, 5, seed=3)
    c = gen.erdos_renyi(100, 80, 5, seed=4)
    assert np.array_equal(a.col, b.col) and np.array_equal(a.val, b.val)
    assert not np.array_equal(a.col, c.col)
    assert np.array_equal(gen.features(10, 4, 1), gen.features(10, 4, 1))
    assert not np.array_equal(gen.features(10, 4, 1), gen.features(10, 4, 2))


def test_erdos_renyi_full_size():
    g = gen.config(1)
    _check_csr(g)
    assert g.M == g.K == 2048 and g.nnz == 16384
    assert np.all(g.degrees() == 8)
    assert g.val.min() >= 0 and g.val.max() < 1


def test_knn_local_small_and_window():
    g = gen.knn_local(M=5000, deg=10, window=512, seed=1)
    _check_csr(g)
    rows = np.repeat(np.arange(g.M), g.degrees())
    assert np.all(g.degrees() == 10) and g.val is None
    assert np.all(np.abs(g.col - rows) <= 512) and np.all(g.col != rows)


@pytest.mark.slow
def test_knn_full_size():
    g = gen.config(2)
    _check_csr(g)
    assert g.M == 1 << 20 and g.nnz == 10 * (1 << 20) and g.val is None


def test_community_structure():
    g = gen.community(n_comm=16, comm_size=64, p=0.2, n_inter=5, seed=2)
    _check_csr(g)
    rows = np.repeat(np.arange(g.M), g.degrees())
    same = (rows // 64) == (g.col // 64)
    n_out = np.bincount(rows[~same], minlength=g.M)
    assert np.all(n_out == 5)
    assert np.all(g.col[same] != rows[same])
    n_in = np.bincount(rows[same], minlength=g.M)
    # Bernoulli(0.2) over 63 members: mean 12.6, sd 3.2; the sample mean of 1024 rows
    assert abs(n_in.mean() - 0.2 * 63) < 5 * np.sqrt(63 * 0.2 * 0.8 / g.M)


def test_community_full_size_degree():
    g = gen.config(4)
    _check_csr(g)
    assert g.M == 65536
    assert abs(g.nnz / g.M - (0.2 * 255 + 5)) < 0.2          # about 56 per row


def test_rmat_small():
    g = gen.rmat(scale=12, edge_factor=16, seed=1)
    _check_csr(g)
    deg = g.degrees()
    nz = deg > 0
    # val = 1/deg(row) after de-duplication
    assert np.array_equal(g.val, np.repeat((1.0 / deg[nz]).astype(np.float32), deg[nz]))
    assert g.nnz <= 16 * 4096 and deg.max() > 20 * deg.mean()      # skewed


def test_chung_lu_small():
    g = gen.chung_lu(M=1 << 14, gamma=2.1, mean=25.0, cap=400.0, seed=3)
    _check_csr(g)
    w = gen.chung_lu_weights(1 << 14, 2.1, 25.0, 400.0)
    assert abs(w.mean() - 25.0) < 1e-6 and w.max() <= 400.0
    assert abs(g.nnz / g.M - 25.0) < 1.0
    assert g.degrees().max() > 200


def test_chung_lu_weights_full_size():
    w = gen.chung_lu_weights(1 << 22, 2.1, 25.0, 1e5)
    assert abs(w.sum() - 25.0 * (1 << 22)) < 1e-3 * (1 << 22)
    assert int((w >= 1e5).sum()) == 50
