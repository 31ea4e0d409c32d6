"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small cases span several tiles, ragged N and forced families / splits; the
edge cases follow the graph-spmm model card ("Correctness"). Full-size
workloads live in test_gpu_workloads.py.
"""
import numpy as np
import pytest

import gen
import oracle
from parity_util import compare, gpu_reduce, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


SMALL = {
    "er": lambda: gen.erdos_renyi(3000, 2500, 8, seed=1),
    "knn": lambda: gen.knn_local(20000, 10, 512, seed=1),
    "knn_weighted": lambda: gen.knn_local(5000, 7, 64, seed=2, weighted=True),
    "rmat": lambda: gen.rmat(scale=13, edge_factor=16, seed=1),
    "community": lambda: gen.community(32, 256, 0.2, 5, seed=1),
    "chung_lu": lambda: gen.chung_lu(1 << 15, 2.1, 25.0, 2000.0, seed=1),
}
_cache = {}


def small(name):
    if name not in _cache:
        _cache[name] = SMALL[name]()
    return _cache[name]


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("N", [1, 3, 16, 17, 32, 64, 130, 256])
def test_small_all_reductions(sdm, cuda_device, name, N):
    g = small(name)
    B = gen.features(g.K, N, seed=N)
    adj = make_adj(sdm, g, cuda_device)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"{name} N={N} {red}")


@pytest.mark.parametrize("family", ["rowgroup", "warprow"])
@pytest.mark.parametrize("t_split", [0, 8, 40])
@pytest.mark.parametrize("N", [4, 16, 36, 64, 128])
def test_forced_families_and_splits(sdm, cuda_device, family, t_split, N):
    g = small("rmat")
    B = gen.features(g.K, N, seed=7)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family(family, t_split)
    info = adj.describe(N)
    assert info["family_name"] == family or info["col_tiles"] > 1
    if t_split:
        assert info["t_split"] == t_split and info["n_heavy"] > 0
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"{family} t={t_split} N={N} {red}")


@pytest.mark.parametrize("family", ["rowgroup", "warprow"])
def test_split_threshold_beyond_int32(sdm, cuda_device, family):
    """A threshold above INT32_MAX splits nothing; every row is still written."""
    g = small("rmat")
    B = gen.features(g.K, 16, seed=8)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family(family, 1 << 40)
    info = adj.describe(16)
    assert info["t_split"] == 2**31 - 1 and info["n_heavy"] == 0
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"{family} t=2^40 {red}")


@pytest.mark.parametrize("t_split", [0, 24])
@pytest.mark.parametrize("N", [128, 132, 256, 384, 520, 1040])
def test_coltile_family(sdm, cuda_device, t_split, N):
    """COLTILE (wide N): staged col/val, bulk copies for long aligned segments,
    padding between rows, tiles beyond N, split rows, ragged N (scalar fallback)."""
    g = small("rmat")
    B = gen.features(g.K, N, seed=N + 5)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("coltile", t_split)
    info = adj.describe(N)
    assert info["family_name"] == ("coltile" if N % 4 == 0 else "warprow")
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"coltile t={t_split} N={N} {red}")
    sdm.spmm_plan_sync(adj.plan)


def test_coltile_unaligned_col_and_long_rows(sdm, cuda_device):
    import torch
    g = small("chung_lu")                          # rows up to thousands of entries
    B = gen.features(g.K, 256, seed=17)
    Bd = to_dev(B, cuda_device)
    for aligned in (True, False):
        if aligned:
            adj = make_adj(sdm, g, cuda_device)
        else:
            cb = torch.empty(g.nnz + 1, dtype=torch.int32, device=cuda_device)
            vb = torch.empty(g.nnz + 1, dtype=torch.float32, device=cuda_device)
            cb[1:].copy_(to_dev(g.col, cuda_device))
            vb[1:].copy_(to_dev(g.val, cuda_device))
            adj = sdm.SparseAdj(to_dev(g.rowptr, cuda_device), cb[1:], vb[1:], num_cols=g.K)
        adj.set_family("coltile", 4000)            # long light rows: bulk copies, many chunks
        for red in ("sum", "max"):
            C, A = gpu_reduce(adj, Bd, red)
            compare(g, B, red, C, A, label=f"coltile long rows aligned={aligned} {red}")
        sdm.spmm_plan_sync(adj.plan)


@pytest.mark.parametrize("family", ["auto", "rowgroup", "warprow", "coltile"])
@pytest.mark.parametrize("t_split", [0, 16])
def test_bitwise_deterministic(sdm, cuda_device, family, t_split):
    import torch
    g = small("chung_lu")
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family(family, t_split)
    for N in (16, 64, 20):
        Bd = to_dev(gen.features(g.K, N, seed=3), cuda_device)
        for red in ("sum", "mean", "max"):
            r1 = adj.reduce(Bd, red)
            r2 = adj.reduce(Bd, red)
            torch.cuda.synchronize()
            if red == "max":
                assert torch.equal(r1[0].view(torch.int32), r2[0].view(torch.int32))
                assert torch.equal(r1[1], r2[1])
            else:
                assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))


def test_descriptors_match_oracle(sdm, cuda_device):
    for name in sorted(SMALL):
        g = small(name)
        adj = make_adj(sdm, g, cuda_device)
        d = adj.describe(16)
        o = oracle.descriptors(g.rowptr)
        for k in ("M", "nnz", "d_max", "n_empty"):
            assert d[k] == o[k], (name, k)
        assert abs(d["dbar"] - o["dbar"]) <= 1e-12 * max(1.0, o["dbar"])
        assert abs(d["cv"] - o["cv"]) <= 1e-9 * max(1.0, o["cv"])
        deg = g.degrees()
        assert d["n_heavy"] == int((deg > d["t_split"]).sum())
        assert d["n_chunks"] == int(np.sum(np.ceil(deg[deg > d["t_split"]] / d["chunk"])))


def test_edge_semantics(sdm, cuda_device):
    """Duplicates summed, unsorted rows, empty rows, ties to the smallest column,
    signed zeros, val=None == all ones (model card, "Correctness")."""
    import json, os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_4x3.json")))
    g = gen.Graph("hand", fx["M"], fx["K"], np.array(fx["rowptr"], np.int32),
                  np.array(fx["col"], np.int32), np.array(fx["val"], np.float32))
    B = np.array(fx["B"], np.float32)
    adj = make_adj(sdm, g, cuda_device)
    Bd = to_dev(B, cuda_device)
    C, _ = gpu_reduce(adj, Bd, "sum")
    assert np.array_equal(C, np.array(fx["sum"], np.float32))
    C, A = gpu_reduce(adj, Bd, "max")
    assert np.array_equal(C.view(np.int32), np.array(fx["max"], np.float32).view(np.int32))
    assert np.array_equal(A, np.array(fx["argmax"], np.int32))
    # unsorted rows with ties and duplicates; constant B -> smallest column
    rows = [[9, 4, 7, 4], [3], [], [8, 1, 1], list(range(99, -1, -1))]
    g = gen.from_rows("u", 5, 100, rows)
    B = np.full((100, 8), 2.5, np.float32)
    adj = make_adj(sdm, g, cuda_device)
    for t_split in (0, 4):
        adj.set_family("auto", t_split)
        C, A = gpu_reduce(adj, to_dev(B, cuda_device), "max")
        assert np.array_equal(A[:, 0], [4, 3, -1, 1, 0])
        compare(g, B, "max", C, A)
    # unweighted == all-ones
    g = small("knn")
    ones = gen.Graph(g.name, g.M, g.K, g.rowptr, g.col, np.ones(g.nnz, np.float32))
    B = gen.features(g.K, 24, seed=9)
    a0, a1 = make_adj(sdm, g, cuda_device), make_adj(sdm, ones, cuda_device)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        c0, x0 = gpu_reduce(a0, Bd, red)
        c1, x1 = gpu_reduce(a1, Bd, red)
        compare(g, B, red, c0, x0)
        compare(ones, B, red, c1, x1)
        if red == "max":
            assert np.array_equal(c0, c1) and np.array_equal(x0, x1)


def test_empty_and_degenerate_shapes(sdm, cuda_device):
    import torch
    # M = 0
    adj = sdm.SparseAdj(torch.zeros(1, dtype=torch.int32, device=cuda_device),
                        torch.zeros(0, dtype=torch.int32, device=cuda_device), num_cols=5)
    n0 = sdm.spmm_launch_count()
    C = adj.reduce(torch.zeros((5, 8), device=cuda_device), "sum")
    assert C.shape == (0, 8) and sdm.spmm_launch_count() == n0
    # nnz = 0: every row empty
    g = gen.from_rows("empty", 40, 7, [[] for _ in range(40)])
    adj = make_adj(sdm, g, cuda_device)
    B = gen.features(7, 12, seed=1)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, to_dev(B, cuda_device), red)
        assert np.all(C == 0)
        if red == "max":
            assert np.all(A == -1)
    # N = 0
    g = small("er")
    adj = make_adj(sdm, g, cuda_device)
    C = adj.reduce(torch.zeros((g.K, 0), device=cuda_device), "sum")
    assert C.shape == (g.M, 0)


def test_single_long_row(sdm, cuda_device):
    rng = np.random.default_rng(3)
    K = 200_000
    cols = np.sort(rng.choice(K, size=100_000, replace=False))
    rows = [[], cols.tolist(), [5, 6]]
    vals = [[], rng.random(100_000).astype(np.float32).tolist(), [1.0, -1.0]]
    g = gen.from_rows("long", 3, K, rows, vals)
    adj = make_adj(sdm, g, cuda_device)
    assert adj.describe(32)["n_heavy"] == 1
    for N in (32, 8, 5):
        B = gen.features(K, N, seed=N)
        Bd = to_dev(B, cuda_device)
        for red in ("sum", "mean", "max"):
            C, A = gpu_reduce(adj, Bd, red)
            compare(g, B, red, C, A, label=f"long row N={N} {red}")


def test_unaligned_pointers_take_scalar_path(sdm, cuda_device):
    import torch
    g = small("er")
    N = 16
    B = gen.features(g.K, N, seed=4)
    adj = make_adj(sdm, g, cuda_device)
    buf = torch.empty(g.K * N + 1, dtype=torch.float32, device=cuda_device)
    Bd = buf[1:].view(g.K, N)
    Bd.copy_(to_dev(B, cuda_device))
    cbuf = torch.empty(g.M * N + 3, dtype=torch.float32, device=cuda_device)
    Cd = cbuf[3:].view(g.M, N)
    for red in ("sum", "mean"):
        adj.reduce(Bd, red, out=Cd)
        torch.cuda.synchronize()
        compare(g, B, red, Cd.cpu().numpy(), None, label=f"unaligned {red}")


def test_one_shot_api(sdm, cuda_device):
    g = small("er")
    B = gen.features(g.K, 8, seed=8)
    rp, cl, vl, Bd = (to_dev(x, cuda_device) for x in (g.rowptr, g.col, g.val, B))
    compare(g, B, "sum", sdm.spmm_sum(rp, cl, vl, Bd).cpu().numpy(), None)
    compare(g, B, "mean", sdm.spmm_mean(rp, cl, vl, Bd).cpu().numpy(), None)
    C, A = sdm.spmm_max(rp, cl, vl, Bd)
    compare(g, B, "max", C.cpu().numpy(), A.cpu().numpy())
    compare(g, B, "sum", (make_adj(sdm, g, cuda_device) @ Bd).cpu().numpy(), None)


def test_invalid_inputs_are_rejected(sdm, cuda_device):
    import torch
    dev = cuda_device
    bad_rowptr = torch.tensor([0, 3, 2, 4], dtype=torch.int32, device=dev)     # decreases
    with pytest.raises(sdm.SpmmError) as e:
        sdm.SparseAdj(bad_rowptr, torch.zeros(4, dtype=torch.int32, device=dev))
    assert e.value.status == 2
    bad0 = torch.tensor([1, 3, 4], dtype=torch.int32, device=dev)             # rowptr[0] != 0
    with pytest.raises(sdm.SpmmError) as e:
        sdm.SparseAdj(bad0, torch.zeros(3, dtype=torch.int32, device=dev))
    assert e.value.status == 2
    rp = torch.tensor([0, 2, 3], dtype=torch.int32, device=dev)
    col = torch.tensor([0, 9, 1], dtype=torch.int32, device=dev)              # 9 >= K = 4
    with pytest.raises(sdm.SpmmError) as e:
        sdm.SparseAdj(rp, col, num_cols=4)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        sdm.SparseAdj(rp, col[:2], num_cols=10)                                # nnz mismatch


def test_allocation_failure_is_reported(sdm, cuda_device, monkeypatch):
    g = small("rmat")
    for n in (1, 2, 3):
        monkeypatch.setenv("SPMM_FAULT_ALLOC", str(n))
        with pytest.raises(sdm.SpmmError) as e:
            make_adj(sdm, g, cuda_device, validate=False)
        assert e.value.status == 3
    monkeypatch.delenv("SPMM_FAULT_ALLOC")
    adj = make_adj(sdm, g, cuda_device)
    B = gen.features(g.K, 16, seed=1)
    C, _ = gpu_reduce(adj, to_dev(B, cuda_device), "sum")
    compare(g, B, "sum", C, None)


# ------------------------------------------------------------- WINDOW family
def _banded_with_extras(M=20001, deg=10, window=64, seed=5):
    """kNN-style band plus: 2 far-away columns on every 7th row (outside any
    window), a block of long rows (overflows the staged entries of their
    tile) and one row long enough to be split."""
    g = gen.knn_local(M, deg, window, seed=seed, weighted=True)
    rng = np.random.default_rng(seed)
    rows = [list(g.col[g.rowptr[i]:g.rowptr[i + 1]]) for i in range(M)]
    vals = [list(g.val[g.rowptr[i]:g.rowptr[i + 1]]) for i in range(M)]
    for i in range(0, M, 7):
        far = rng.integers(0, M, size=2).tolist()
        rows[i] += far
        vals[i] += rng.random(2).astype(np.float32).tolist()
    for i in range(5000, 5100):
        lo, hi = max(0, i - window), min(M, i + window + 1)
        extra = rng.integers(lo, hi, size=100).tolist()
        rows[i] += extra
        vals[i] += rng.random(100).astype(np.float32).tolist()
    rows[9000] = rng.integers(0, M, size=3001).tolist()
    vals[9000] = rng.random(3001).astype(np.float32).tolist()
    return gen.from_rows("banded_extras", M, M, rows, vals)


@pytest.mark.parametrize("N", [4, 8, 16, 20, 32, 48, 64, 128, 256])
def test_window_family_banded(sdm, cuda_device, N):
    g = small("knn")
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("window")
    info = adj.describe(N)
    assert info["family_name"] == "window", info
    assert info["band_w"] == 512
    B = gen.features(g.K, N, seed=N + 100)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"window knn N={N} {red}")
    sdm.spmm_plan_sync(adj.plan)


@pytest.mark.parametrize("N", [16, 36, 64, 128])
def test_window_family_irregular(sdm, cuda_device, N):
    g = _banded_with_extras()
    assert g.nnz % 4 != 0
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("window")
    info = adj.describe(N)
    assert info["family_name"] == "window" and info["n_heavy"] == 1, info
    B = gen.features(g.K, N, seed=N + 200)
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"window irregular N={N} {red}")
    sdm.spmm_plan_sync(adj.plan)
    # deterministic
    import torch
    r1, r2 = adj.reduce(Bd, "sum"), adj.reduce(Bd, "sum")
    torch.cuda.synchronize()
    assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))


def test_window_family_community_and_unaligned_col(sdm, cuda_device):
    import torch
    g = small("community")
    adj = make_adj(sdm, g, cuda_device)
    assert adj.describe(64)["band_w"] == 256
    adj.set_family("window")
    B = gen.features(g.K, 64, seed=3)
    Bd = to_dev(B, cuda_device)
    assert adj.describe(64)["family_name"] == "window"
    for red in ("sum", "max"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"window community {red}")
    # col/val views that are not 16-byte aligned: the router must avoid WINDOW
    cbuf = torch.empty(g.nnz + 1, dtype=torch.int32, device=cuda_device)
    vbuf = torch.empty(g.nnz + 1, dtype=torch.float32, device=cuda_device)
    cbuf[1:].copy_(to_dev(g.col, cuda_device))
    vbuf[1:].copy_(to_dev(g.val, cuda_device))
    adj2 = sdm.SparseAdj(to_dev(g.rowptr, cuda_device), cbuf[1:], vbuf[1:], num_cols=g.K)
    adj2.set_family("window")
    C, A = gpu_reduce(adj2, Bd, "sum")
    compare(g, B, "sum", C, A, label="window unaligned col")


def test_bounded_wait_reports_timeout_and_context_survives(sdm, cuda_device):
    """A wait that nothing completes gives up after its limit: the plan reports
    SPMM_ERR_TIMEOUT (6), the error words are cleared, and the plan and the
    context keep working."""
    g = small("er")
    adj = make_adj(sdm, g, cuda_device)
    assert sdm.spmm_check_wait_timeout(adj.plan, 2000) == 6
    sdm.spmm_plan_sync(adj.plan)                    # cleared: no error left behind
    B = gen.features(g.K, 16, seed=1)
    C, A = gpu_reduce(adj, to_dev(B, cuda_device), "sum")
    compare(g, B, "sum", C, A, label="after a timeout")
    adj.close()
