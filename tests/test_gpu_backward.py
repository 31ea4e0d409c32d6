"""Backward path on the GPU vs the oracle, through the C ABI.

* spmm_transpose: rowptrT, colT and valT bit-identical to the oracle's stable
  transpose (scaled mean values too: both sides divide in fp64 and round once).
* sum / mean backward: a product with the GPU transpose, held to the forward's
  tolerance 1e-5 * T + 1e-6 against the oracle's product with its own transpose.
* max-pool backward: 1e-5 * T + 1e-6 with T = max |a| times the sum of
  |dC[i, c]| over the rows that chose column j. Duplicated pairs pass the
  gradient through the one copy whose product won (weighted copies differ; a
  run of copies can straddle a chunk boundary of a split row). The argmax fed
  to both sides is the oracle's; the GPU's forward argmax is first checked equal.
"""
import numpy as np
import pytest

import gen
import oracle
from parity_util import ATOL, RTOL, compare, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


def dup_graph(seed, M=3000, K=700, weighted=True):
    """Random rows with duplicated pairs and empty rows."""
    rng = np.random.default_rng(seed)
    rows, vals = [], []
    for i in range(M):
        d = 0 if rng.random() < 0.1 else int(rng.integers(1, 40))
        c = rng.integers(0, K, size=d).tolist()
        if d >= 2 and rng.random() < 0.3:
            c[-1] = c[0]
        rows.append(c)
        vals.append(rng.standard_normal(d).astype(np.float32).tolist())
    return gen.from_rows(f"dup{seed}", M, K, rows, vals if weighted else None)


GRAPHS = {
    "er": lambda: gen.erdos_renyi(3000, 2500, 8, seed=1),
    "knn_weighted": lambda: gen.knn_local(20000, 7, 64, seed=2, weighted=True),
    "rmat": lambda: gen.rmat(scale=13, edge_factor=16, seed=1),
    "chung_lu": lambda: gen.chung_lu(1 << 15, 2.1, 25.0, 2000.0, seed=1),
    "dup": lambda: dup_graph(3),
    "dup_unweighted": lambda: dup_graph(4, weighted=False),
    "k1": lambda: gen.from_rows("k1", 5000, 1, [[0] * (i % 4) for i in range(5000)]),
    "k256": lambda: gen.erdos_renyi(9000, 256, 5, seed=5),       # one radix pass
    "k257": lambda: gen.erdos_renyi(9000, 257, 5, seed=6),       # two passes
    "k70000": lambda: gen.erdos_renyi(3000, 70000, 9, seed=7),   # three passes
    "empty": lambda: gen.from_rows("empty", 50, 40, [[] for _ in range(50)]),
    "hub": lambda: hub_graph(),
}


def hub_graph(M=6000, K=900):
    """Every row holds column 7 (a row of 6000 entries in A^T, split into
    chunks) plus a few random columns; some rows repeat column 7."""
    rng = np.random.default_rng(9)
    rows, vals = [], []
    for i in range(M):
        c = [7] + rng.integers(0, K, size=int(rng.integers(0, 6))).tolist()
        if i % 11 == 0:
            c.append(7)
        rng.shuffle(c)
        rows.append(c)
        vals.append(rng.standard_normal(len(c)).astype(np.float32).tolist())
    return gen.from_rows("hub", M, K, rows, vals)


_cache = {}


def graph(name):
    if name not in _cache:
        _cache[name] = GRAPHS[name]()
    return _cache[name]


def gpu_transpose(adj, scale_mean):
    import torch
    t = adj.transpose(scale_mean=scale_mean)
    torch.cuda.synchronize()
    return t, (t.rowptr.cpu().numpy(), t.col.cpu().numpy(),
               None if t.val is None else t.val.cpu().numpy())


@pytest.mark.parametrize("name", sorted(GRAPHS))
@pytest.mark.parametrize("scale_mean", [False, True])
def test_transpose_bit_exact(sdm, cuda_device, name, scale_mean):
    g = graph(name)
    adj = make_adj(sdm, g, cuda_device)
    t, (rT, cT, vT) = gpu_transpose(adj, scale_mean)
    oR, oC, oV = oracle.transpose(g.rowptr, g.col, g.val, g.K, scale_mean=scale_mean)
    assert t.M == g.K and t.K == g.M
    assert np.array_equal(rT, oR)
    assert np.array_equal(cT, oC)
    if oV is None:
        assert vT is None
    else:
        assert vT is not None and np.array_equal(vT.view(np.int32), oV.view(np.int32))
    t.close()
    adj.close()


def test_transpose_is_deterministic(sdm, cuda_device):
    g = graph("chung_lu")
    adj = make_adj(sdm, g, cuda_device)
    _, a = gpu_transpose(adj, True)
    _, b = gpu_transpose(adj, True)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.int32), y.view(np.int32))


@pytest.mark.parametrize("name", ["er", "knn_weighted", "rmat", "chung_lu", "dup",
                                  "dup_unweighted", "k1", "empty"])
@pytest.mark.parametrize("N", [1, 16, 33, 64])
def test_sum_and_mean_backward(sdm, cuda_device, name, N):
    import torch
    g = graph(name)
    dC = gen.features(g.M, N, seed=11, tag="dC")
    adj = make_adj(sdm, g, cuda_device)
    dCd = to_dev(dC, cuda_device)
    for red, scale in (("sum", False), ("mean", True)):
        got = adj.backward(dCd, red)
        torch.cuda.synchronize()
        oR, oC, oV = oracle.transpose(g.rowptr, g.col, g.val, g.K, scale_mean=scale)
        gT = gen.Graph(g.name + "^T", g.K, g.M, oR, oC, oV)
        compare(gT, dC, "sum", got.cpu().numpy(), None, label=f"{name} N={N} {red} backward")
    adj.close()


def check_maxpool(sdm, dev, g, N, seed=0):
    import torch
    B = gen.features(g.K, N, seed=seed)
    dC = gen.features(g.M, N, seed=seed + 1, tag="dC")
    adj = make_adj(sdm, g, dev)
    C, A = adj.reduce(to_dev(B, dev), "max")
    torch.cuda.synchronize()
    _, Ar, _ = oracle.spmm(g.rowptr, g.col, g.val, B, "max")
    assert np.array_equal(A.cpu().numpy(), Ar)
    got = adj.backward(to_dev(dC, dev), "max", argmax=to_dev(Ar, dev),
                       B=None if g.val is None else to_dev(B, dev))
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    want = oracle.maxpool_backward(g.rowptr, g.col, g.val, Ar, dC, g.K, B)
    # scale of the tolerance: max |a| times the sum of |dC[i, c]| over the rows
    # that chose j (a bound of the sum of |a_w * dC[i, c]|)
    amax = 1.0 if g.val is None or g.nnz == 0 else float(np.abs(g.val).max())
    T = oracle.maxpool_backward(g.rowptr, g.col, None, Ar, np.abs(dC), g.K) * amax
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bound = RTOL * T.astype(np.float64) + ATOL
    assert not (err > bound).any(), f"{g.name} N={N}: {int((err > bound).sum())} outside tolerance"
    # columns no row chose are exactly zero
    assert np.all(got[T == 0] == 0)
    adj.close()
    return got


@pytest.mark.parametrize("name", ["er", "knn_weighted", "rmat", "chung_lu", "dup",
                                  "dup_unweighted", "k1", "empty", "hub"])
@pytest.mark.parametrize("N", [1, 16, 33, 64, 130])
def test_maxpool_backward(sdm, cuda_device, name, N):
    check_maxpool(sdm, cuda_device, graph(name), N)


def test_maxpool_backward_split_rows(sdm, cuda_device):
    """The hub column's row of A^T exceeds the split threshold."""
    g = graph("hub")
    adj = make_adj(sdm, g, cuda_device)
    t = adj.transpose()
    assert t.describe(16)["n_heavy"] >= 1
    t.close()
    adj.close()
    check_maxpool(sdm, cuda_device, g, 16)


def test_maxpool_backward_duplicates_across_chunks(sdm, cuda_device):
    """Copies of one pair (i, 7) placed so that every chunk boundary of the
    split row 7 of A^T falls inside a run of copies (runs of 3 copies with
    distinct weights): each run must count once, in the chunk where it starts."""
    M, K = 4000, 50
    rng = np.random.default_rng(21)
    rows = [[7, 7, 7] + rng.integers(0, K, size=2).tolist() for _ in range(M)]
    vals = [rng.standard_normal(len(r)).astype(np.float32).tolist() for r in rows]
    g = gen.from_rows("runs", M, K, rows, vals)
    adj = make_adj(sdm, g, cuda_device)
    t = adj.transpose()
    info = t.describe(16)
    assert info["n_heavy"] >= 1 and info["chunk"] % 3 != 0
    t.close()
    adj.close()
    check_maxpool(sdm, cuda_device, g, 16)
    check_maxpool(sdm, cuda_device, gen.from_rows("runs_u", M, K, rows, None), 16)


def test_maxpool_backward_deterministic(sdm, cuda_device):
    a = check_maxpool(sdm, cuda_device, graph("rmat"), 64)
    b = check_maxpool(sdm, cuda_device, graph("rmat"), 64)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


def test_transpose_full_size_knn(sdm, cuda_device):
    """The 1M-row kNN workload (10M entries): the whole transpose, bit-exact."""
    g = gen.config(2)
    adj = make_adj(sdm, g, cuda_device)
    t, (rT, cT, vT) = gpu_transpose(adj, True)
    oR, oC, oV = oracle.transpose(g.rowptr, g.col, g.val, g.K, scale_mean=True)
    assert np.array_equal(rT, oR) and np.array_equal(cT, oC)
    assert np.array_equal(vT.view(np.int32), oV.view(np.int32))
    t.close()
    adj.close()


def test_backward_invalid_args(sdm, cuda_device):
    g = graph("er")
    adj = make_adj(sdm, g, cuda_device)
    with pytest.raises(sdm.SpmmError):
        sdm.spmm_transpose(adj.plan, adj.col.data_ptr(), None, False, None, None, None)
    with pytest.raises(ValueError):
        adj.backward(to_dev(gen.features(g.M, 4, seed=1), cuda_device), "max")
    adj.close()
