"""BLOCK family (tensor cores, split TF32) vs the oracle.

Sum and mean within 1e-5 * T + 1e-6 (T from the oracle); forced and routed;
unweighted (two MMA passes) and weighted (three); rows unsorted (the scan
path), partial row tiles and column tiles, long rows, the fused epilogue.
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


def irregular_blocks(M=1000, K=1100, seed=3, weighted=True, shuffle=False, long_row=None):
    """Entries mostly inside the 256-column diagonal blocks, some outside,
    duplicates, empty rows; M and K not multiples of the tile sizes."""
    rng = np.random.default_rng(seed)
    rows, vals = [], []
    for i in range(M):
        b0 = i // 256 * 256
        d = 0 if rng.random() < 0.05 else int(rng.integers(1, 60))
        c = rng.integers(b0, min(b0 + 256, K), size=d).tolist()
        c += rng.integers(0, K, size=int(rng.integers(0, 4))).tolist()
        if len(c) > 2 and rng.random() < 0.2:
            c.append(c[0])
        if i == long_row:
            c += rng.integers(0, K, size=3000).tolist()
        c = sorted(c) if not shuffle else rng.permutation(c).tolist()
        rows.append(c)
        vals.append((rng.random(len(c)) * 2 - 1).astype(np.float32).tolist())
    return gen.from_rows("blocks", M, K, rows, vals if weighted else None)


_cache = {}


def unweighted(g):
    return gen.Graph(g.name + "_unweighted", g.M, g.K, g.rowptr, g.col, None)


def graph(name):
    if name not in _cache:
        _cache[name] = {
            "community": lambda: gen.community(32, 256, 0.2, 5, seed=1),
            "community_unweighted": lambda: unweighted(gen.community(16, 256, 0.2, 5, seed=2)),
            "irregular": lambda: irregular_blocks(),
            "irregular_unweighted": lambda: irregular_blocks(seed=4, weighted=False),
            "unsorted": lambda: irregular_blocks(seed=5, shuffle=True),
            "long_row": lambda: irregular_blocks(seed=6, long_row=77),
        }[name]()
    return _cache[name]


@pytest.mark.parametrize("name", ["community", "community_unweighted", "irregular",
                                  "irregular_unweighted", "unsorted", "long_row"])
@pytest.mark.parametrize("N", [16, 48, 128, 144, 256])
def test_block_forced(sdm, cuda_device, name, N):
    g = graph(name)
    B = gen.features(g.K, N, seed=N + 11)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("block")
    Bd = to_dev(B, cuda_device)
    for red in ("sum", "mean"):
        assert adj.describe(N, red)["family_name"] == "block"
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, label=f"block {name} N={N} {red}")
    sdm.spmm_plan_sync(adj.plan)
    adj.close()


def test_block_descriptors_and_pinning(sdm, cuda_device):
    g = graph("community")
    adj = make_adj(sdm, g, cuda_device)
    info = adj.describe(128, "sum")
    assert info["rows_sorted"] == 1 and info["blk_intra"] > 0.85 * g.nnz
    assert info["family_name"] == "block"                          # routed
    assert info["block_bytes"] == 0                                 # prepared on first use
    adj.set_family("warprow")
    assert adj.describe(128, "sum")["family_name"] == "warprow"
    adj.set_family("block")
    info = adj.describe(128, "sum")
    assert info["family_name"] == "block" and info["launches"] == 1
    assert adj.describe(128, "max")["family_name"] != "block"
    assert adj.describe(20, "sum")["family_name"] != "block"       # N % 16 != 0
    B = gen.features(g.K, 128, seed=5)
    C, A = gpu_reduce(adj, to_dev(B, cuda_device), "max")
    compare(g, B, "max", C, A, label="community max (SIMT)")
    # preparation: explicit, then reported; 256 KB per 128-row tile + the
    # compact CSR of the entries outside the diagonal blocks
    sdm.spmm_plan_prepare_blocks(adj.plan, adj.col.data_ptr(), adj.val.data_ptr())
    n_off = g.nnz - info["blk_intra"]
    want = (g.M + 127) // 128 * 256 * 1024 + 4 * (g.M + 1) + 8 * n_off
    assert adj.describe(128, "sum")["block_bytes"] == want
    C, A = gpu_reduce(adj, to_dev(B, cuda_device), "sum")
    compare(g, B, "sum", C, A, label="community sum after explicit preparation")
    adj.close()


def test_block_reprepares_for_the_other_flavour(sdm, cuda_device):
    """The prepared pieces belong to one flavour of A (weighted or not): a run
    with the other flavour prepares again, and every run stays correct."""
    import torch
    g = graph("community")
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("block")
    N = 64
    B = gen.features(g.K, N, seed=6)
    Bd = to_dev(B, cuda_device)
    Cd = torch.empty((g.M, N), dtype=torch.float32, device=cuda_device)
    for weighted in (True, False, True):
        gg = g if weighted else unweighted(g)
        sdm.spmm_run(adj.plan, adj.col.data_ptr(), adj.val.data_ptr() if weighted else None,
                     Bd.data_ptr(), N, sdm.REDUCE["sum"], Cd.data_ptr())
        torch.cuda.synchronize()
        compare(gg, B, "sum", Cd.cpu().numpy(), None,
                label=f"block {'weighted' if weighted else 'unweighted'}")
    adj.close()


def test_block_deterministic_and_epilogue(sdm, cuda_device):
    import torch
    g = graph("irregular")
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("block")
    N = 64
    B = gen.features(g.K, N, seed=9)
    bias = gen.features(1, N, seed=10)[0]
    Bd, bd = to_dev(B, cuda_device), to_dev(bias, cuda_device)
    r1 = adj.reduce(Bd, "sum", bias=bd, activation="relu")
    r2 = adj.reduce(Bd, "sum", bias=bd, activation="relu")
    torch.cuda.synchronize()
    assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))
    Cr, _, Tr = oracle.spmm(g.rowptr, g.col, g.val, B, "sum", bias=bias, act="relu")
    T = Tr.astype(np.float64) + np.abs(bias.astype(np.float64))
    err = np.abs(r1.cpu().numpy().astype(np.float64) - Cr.astype(np.float64))
    assert not (err > 1e-5 * T + 1e-6).any()
    adj.close()
