"""STREAM family (equal entry ranges per lane group, SIMT gathers with the
next batch's columns, values and row ids loaded ahead) against the oracle,
pinned with spmm_plan_set_family, through the C ABI.

The cases put rows across every boundary the family has: a row that spans
several batches of a range, rows cut by the ranges (combined by the second
launch), one row long enough to span many ranges, runs of empty rows
(inside a range, between two ranges, before the first and after the last
entry), graphs with few entries (ranges of 16), unsorted and duplicated
entries, both lane shapes (16 lanes up to N = 64, else 32 lanes per
128-column tile) with idle lanes and ragged last tiles, the fused epilogue,
row-range plans, and bitwise reproducibility. Tolerance and bit-exactness as
in every parity test.
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
    """Row 1234 holds 400,000 entries (many ranges); the others 0-12
    random entries, some rows empty."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(M):
        d = long_len if i == 1234 else int(rng.integers(0, 13))
        rows.append(rng.integers(0, K, size=d).tolist())
    vals = [rng.standard_normal(len(r)).astype(np.float32).tolist() for r in rows]
    return gen.from_rows("long_row", M, K, rows, vals)


def empty_runs_graph(M=60000, K=700, seed=4):
    """Long runs of empty rows between short rows (some longer than a CTA's
    range of entries), empty rows first and last, unsorted columns and
    duplicated pairs."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(M):
        if i < 50 or i >= M - 70 or (i // 2000) % 2 == 1 or rng.random() < 0.3:
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
    "long_row": long_row_graph,
    "empty_runs": empty_runs_graph,
    # few entries: one range, or a few of 16
    "tiny": lambda: gen.from_rows("tiny", 5, 9, [[1, 3], [], [8, 8, 0], [], [2]],
                                  [[0.5, -1.0], [], [2.0, 3.0, -4.0], [], [1.5]]),
    "one_entry": lambda: gen.from_rows("one_entry", 40, 3, [[] if i != 17 else [2]
                                                            for i in range(40)],
                                       [[] if i != 17 else [-2.5] for i in range(40)]),
}
_cache = {}


def graph(name):
    if name not in _cache:
        _cache[name] = GRAPHS[name]()
    return _cache[name]


def stream_adj(sdm, g, dev, N, red, rows=None):
    if rows is None:
        adj = make_adj(sdm, g, dev)
    else:
        adj = sdm.SparseAdj(to_dev(g.rowptr, dev), to_dev(g.col, dev),
                            None if g.val is None else to_dev(g.val, dev), num_cols=g.K,
                            rows=rows)
    adj.set_family("stream")
    info = adj.describe(N, red)
    assert info["family_name"] == "stream", info
    return adj, info


@pytest.mark.parametrize("name", sorted(GRAPHS))
@pytest.mark.parametrize("N", [48, 64, 128, 256])
def test_stream_all_reductions(sdm, cuda_device, name, N):
    g = graph(name)
    B = gen.features(g.K, N, seed=N + 3)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        adj, info = stream_adj(sdm, g, cuda_device, N, red)
        assert info["lanes"] == (16 if N <= 64 else 32)
        assert 1 <= info["stream_ranges"] <= max(1, g.nnz)
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"stream {name} N={N} {red}")
        adj.close()


@pytest.mark.parametrize("N,tiles", [(260, 3), (512, 4)])
def test_stream_column_tiles(sdm, cuda_device, N, tiles):
    """Three tiles of 128 columns, the last with one active lane; four tiles."""
    for name in ("chung_lu", "long_row"):
        g = graph(name)
        B = gen.features(g.K, N, seed=5)
        Bd = to_dev(B, cuda_device)
        for red in ("sum", "max"):
            adj, info = stream_adj(sdm, g, cuda_device, N, red)
            assert info["col_tiles"] == tiles
            C, A = gpu_reduce(adj, Bd, red)
            compare(g, B, red, C, A, label=f"stream {name} N={N} {red}")
            adj.close()


def test_stream_long_row_spans_ranges(sdm, cuda_device):
    g = graph("long_row")
    adj, info = stream_adj(sdm, g, cuda_device, 256, "sum")
    per_range = g.nnz / info["stream_ranges"]
    assert 400_000 > 10 * per_range, (g.nnz, info["stream_ranges"])
    adj.close()


def test_stream_row_ids_built_once(sdm, cuda_device):
    """The per-entry row ids (4 bytes per entry) appear with the first run."""
    g = graph("rmat")
    B = gen.features(g.K, 64, seed=1)
    Bd = to_dev(B, cuda_device)
    adj, info = stream_adj(sdm, g, cuda_device, 64, "sum")
    assert info["gather_bytes"] == 0
    C1, _ = gpu_reduce(adj, Bd, "sum")
    assert adj.describe(64, "sum")["gather_bytes"] == 4 * g.nnz
    C2, _ = gpu_reduce(adj, Bd, "sum")
    assert np.array_equal(C1.view(np.int32), C2.view(np.int32))
    adj.close()


def test_stream_reserve_builds_row_ids(sdm, cuda_device):
    """spmm_plan_reserve for a product routed to STREAM builds the row ids up
    front, so the first product allocates nothing more."""
    import torch
    g = graph("chung_lu")
    B = gen.features(g.K, 64, seed=4)
    Bd = to_dev(B, cuda_device)
    adj, info = stream_adj(sdm, g, cuda_device, 64, "max")
    assert info["gather_bytes"] == 0
    adj.reserve(64, "max")
    assert adj.describe(64, "max")["gather_bytes"] == 4 * g.nnz
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    C, A = gpu_reduce(adj, Bd, "max")
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)   # outputs only, no workspace
    compare(g, B, "max", C, A, label="stream after reserve")
    adj.close()


def test_stream_epilogue(sdm, cuda_device):
    import torch

    import oracle
    g = graph("chung_lu")
    N = 128
    B = gen.features(g.K, N, seed=9)
    bias = gen.features(1, N, seed=10)[0]
    Bd, bd = to_dev(B, cuda_device), to_dev(bias, cuda_device)
    for red in ("sum", "mean", "max"):
        adj, _ = stream_adj(sdm, g, cuda_device, N, red)
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
def test_stream_bitwise_deterministic(sdm, cuda_device, name):
    g = graph(name)
    B = gen.features(g.K, 256, seed=1)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "max"):
        adj, _ = stream_adj(sdm, g, cuda_device, 256, red)
        C1, A1 = gpu_reduce(adj, Bd, red)
        C2, A2 = gpu_reduce(adj, Bd, red)
        assert np.array_equal(C1.view(np.int32), C2.view(np.int32))
        if red == "max":
            assert np.array_equal(A1, A2)
        adj.close()


def test_stream_row_range_plan(sdm, cuda_device):
    """A plan over rows [b, e) of the arrays: local row ids, the range's
    own entries only."""
    g = graph("chung_lu")
    b, e = 1001, 20017
    B = gen.features(g.K, 256, seed=6)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "max"):
        adj, _ = stream_adj(sdm, g, cuda_device, 256, red, rows=(b, e))
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, rows=np.arange(b, e), label=f"stream range {red}")
        adj.close()


@pytest.mark.parametrize("N,name", [(32, "rmat"), (66, "rmat"), (256, "no_entries")])
def test_stream_falls_back(sdm, cuda_device, N, name):
    """N <= 32, N % 4 != 0, or no entry at all: another family, correctly."""
    g = (gen.from_rows("no_entries", 700, 10, [[] for _ in range(700)])
         if name == "no_entries" else graph(name))
    B = gen.features(g.K, N, seed=2)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("stream")
    assert adj.describe(N, "sum")["family_name"] != "stream"
    for red in ("sum", "max"):
        C, A = gpu_reduce(adj, to_dev(B, cuda_device), red)
        compare(g, B, red, C, A, label=f"stream fallback {name} N={N} {red}")
    adj.close()


_full = {}


@pytest.mark.parametrize("cid,N,red", [(5, 64, "sum"), (5, 64, "max"), (5, 256, "mean"),
                                       (3, 64, "sum"), (3, 256, "max")])
def test_stream_full_size(sdm, cuda_device, cid, N, red):
    """The 4M-row Chung-Lu graph and R-MAT scale 20 at the launch shape the
    bench times: a seeded sample of rows, every row at a range boundary
    (combined by the second launch), and the longest rows."""
    import torch
    if _full.get("cid") != cid:
        _full.clear()
        _full.update(cid=cid, g=gen.config(cid))
    g = _full["g"]
    B = gen.features(g.K, N, seed=0)
    Bd = to_dev(B, cuda_device)
    adj, info = stream_adj(sdm, g, cuda_device, N, red)
    W = info["stream_ranges"]
    cuts = [g.nnz * k // W for k in range(1, W)]
    edge_rows = np.searchsorted(g.rowptr, cuts, side="right") - 1
    deg = np.diff(g.rowptr)
    rng = np.random.default_rng(cid * 1000 + N)
    rows = np.unique(np.concatenate([edge_rows, edge_rows + 1, np.argsort(deg)[-64:],
                                     rng.integers(0, g.M, 20000), [0, g.M - 1]]))
    rows = rows[(rows >= 0) & (rows < g.M)]
    C, A = gpu_reduce(adj, Bd, red, rows=rows)
    compare(g, B, red, C, A, rows=rows, label=f"stream config {cid} N={N} {red}")
    adj.close()
    del Bd
    torch.cuda.empty_cache()
