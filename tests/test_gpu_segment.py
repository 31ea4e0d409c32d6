"""SEGMENT family (merge-path tiles of entries plus row ends) against the
oracle, pinned with spmm_plan_set_family, through the C ABI.

The cases put rows across every boundary the family has: group slices inside
a tile, tiles inside a warp's range (the row carried in registers), and warp
ranges (the partials combined by the second launch), including one row long
enough to span several warp ranges, runs of empty rows, unsorted and
duplicated entries, a graph with fewer tiles than warps, N that needs two
chunks per lane and several column tiles, the fused epilogue, and bitwise
reproducibility. Tolerance and bit-exactness as in every parity test.
"""
import numpy as np
import pytest

import gen
from parity_util import compare, gpu_reduce, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


def long_row_graph(M=3000, K=5000, long_len=400_000, seed=3):
    """Row 1234 holds 400,000 entries (several warp ranges of 544-item tiles
    on a full GPU); the others 0-12 random entries, some rows empty."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(M):
        d = long_len if i == 1234 else int(rng.integers(0, 13))
        rows.append(rng.integers(0, K, size=d).tolist())
    vals = [rng.standard_normal(len(r)).astype(np.float32).tolist() for r in rows]
    return gen.from_rows("long_row", M, K, rows, vals)


def empty_runs_graph(M=60000, K=700, seed=4):
    """Long runs of empty rows (a tile of row ends only) between short rows,
    unsorted columns and duplicated pairs."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(M):
        if (i // 2000) % 2 == 1 or rng.random() < 0.3:
            rows.append([])
            continue
        c = rng.integers(0, K, size=int(rng.integers(1, 30))).tolist()
        if len(c) > 2 and rng.random() < 0.3:
            c.append(c[0])
        rows.append(c)
    vals = [rng.random(len(r)).astype(np.float32).tolist() for r in rows]
    return gen.from_rows("empty_runs", M, K, rows, vals)


def unweighted(g):
    return gen.Graph(g.name + "_u", g.M, g.K, g.rowptr, g.col, None)


GRAPHS = {
    "er": lambda: gen.erdos_renyi(3000, 2500, 8, seed=1),
    "rmat": lambda: gen.rmat(scale=13, edge_factor=16, seed=1),
    "rmat_unweighted": lambda: unweighted(gen.rmat(scale=12, edge_factor=16, seed=2)),
    "chung_lu": lambda: gen.chung_lu(1 << 15, 2.1, 25.0, 2000.0, seed=1),
    "knn": lambda: gen.knn_local(20000, 10, 512, seed=1),
    "community": lambda: gen.community(32, 256, 0.2, 5, seed=1),
    "long_row": long_row_graph,
    "empty_runs": empty_runs_graph,
    "tiny": lambda: gen.from_rows("tiny", 5, 9, [[1, 3], [], [8, 8, 0], [], [2]],
                                  [[0.5, -1.0], [], [2.0, 3.0, -4.0], [], [1.5]]),
    "no_entries": lambda: gen.from_rows("no_entries", 700, 10, [[] for _ in range(700)]),
}
_cache = {}


def graph(name):
    if name not in _cache:
        _cache[name] = GRAPHS[name]()
    return _cache[name]


def segment_adj(sdm, g, dev, N, red):
    adj = make_adj(sdm, g, dev)
    adj.set_family("segment")
    info = adj.describe(N, red)
    assert info["family_name"] == "segment", info
    return adj, info


@pytest.mark.parametrize("name", sorted(GRAPHS))
@pytest.mark.parametrize("N", [4, 16, 64, 128, 132, 256])
def test_segment_all_reductions(sdm, cuda_device, name, N):
    g = graph(name)
    B = gen.features(g.K, N, seed=N + 3)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        adj, info = segment_adj(sdm, g, cuda_device, N, red)
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"segment {name} N={N} {red}")
        adj.close()


@pytest.mark.parametrize("N", [260, 520])
def test_segment_column_tiles(sdm, cuda_device, N):
    """Two chunks per lane and two or three column tiles, the last one ragged."""
    g = graph("chung_lu")
    B = gen.features(g.K, N, seed=5)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "max"):
        adj, info = segment_adj(sdm, g, cuda_device, N, red)
        assert info["seg_chunks"] == 2 and info["col_tiles"] == (N + 255) // 256
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"segment N={N} {red}")
        adj.close()


def test_segment_long_row_spans_warp_ranges(sdm, cuda_device):
    g = graph("long_row")
    adj, info = segment_adj(sdm, g, cuda_device, 16, "sum")
    # the long row alone is several warps' share of the tiles
    per_warp = info["seg_tiles"] / info["seg_warps"] * 544
    assert 400_000 > 3 * per_warp, (info["seg_tiles"], info["seg_warps"])
    adj.close()


def test_segment_epilogue(sdm, cuda_device):
    import torch
    g = graph("chung_lu")
    N = 64
    B = gen.features(g.K, N, seed=9)
    bias = gen.features(1, N, seed=10)[0]
    Bd, bd = to_dev(B, cuda_device), to_dev(bias, cuda_device)
    import oracle
    for red in ("sum", "mean", "max"):
        adj, _ = segment_adj(sdm, g, cuda_device, N, red)
        res = adj.reduce(Bd, red, bias=bd, activation="relu")
        C = (res[0] if red == "max" else res)
        torch.cuda.synchronize()
        Cr, Ar, Tr = oracle.spmm(g.rowptr, g.col, g.val, B, red, bias=bias, act="relu")
        C = C.cpu().numpy()
        if red == "max":
            assert np.array_equal(C.view(np.int32), Cr.view(np.int32))
            assert np.array_equal(res[1].cpu().numpy(), Ar)
        else:
            err = np.abs(C.astype(np.float64) - Cr.astype(np.float64))
            assert np.all(err <= 1e-5 * (Tr + np.abs(bias)[None, :]) + 1e-6), red
        adj.close()


@pytest.mark.parametrize("name", ["long_row", "rmat"])
def test_segment_bitwise_deterministic(sdm, cuda_device, name):
    g = graph(name)
    B = gen.features(g.K, 64, seed=1)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "max"):
        adj, _ = segment_adj(sdm, g, cuda_device, 64, red)
        C1, A1 = gpu_reduce(adj, Bd, red)
        C2, A2 = gpu_reduce(adj, Bd, red)
        assert np.array_equal(C1.view(np.int32), C2.view(np.int32))
        if red == "max":
            assert np.array_equal(A1, A2)
        adj.close()


def test_segment_unaligned_operands_fall_back(sdm, cuda_device):
    """N % 4 != 0 (no 128-bit vectors) is served by another family, correctly."""
    g = graph("rmat")
    B = gen.features(g.K, 6, seed=2)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("segment")
    assert adj.describe(6, "sum")["family_name"] != "segment"
    C, A = gpu_reduce(adj, to_dev(B, cuda_device), "sum")
    compare(g, B, "sum", C, A, label="segment fallback N=6")
    adj.close()


_full = {}


@pytest.mark.parametrize("cid,N,red", [(3, 64, "sum"), (3, 64, "max"), (5, 16, "sum"),
                                       (5, 16, "max")])
def test_segment_full_size(sdm, cuda_device, cid, N, red):
    """R-MAT scale 20 and the 4M-row Chung-Lu graph, every element."""
    import torch
    if _full.get("cid") != cid:
        _full.clear()
        _full.update(cid=cid, g=gen.config(cid))
    g = _full["g"]
    B = gen.features(g.K, N, seed=0)
    Bd = to_dev(B, cuda_device)
    adj, _ = segment_adj(sdm, g, cuda_device, N, red)
    C, A = gpu_reduce(adj, Bd, red)
    compare(g, B, red, C, A, label=f"segment config {cid} N={N} {red}")
    adj.close()
    del Bd
    torch.cuda.empty_cache()
