"""Row-range plans (spmm_plan_create_range) against the oracle on the GPU.

A range plan computes the rows [b, e) of a larger matrix from the whole
matrix's rowptr, col and val. Its outputs must equal the oracle's for those
global rows (max and argmax bit for bit, sum and mean within 1e-5*T + 1e-6),
whichever family it routes to, and the shards of spmm_partition_rows must
reproduce the whole matrix's product.
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


def _range_adj(sdm, g, dev, b, e):
    return sdm.SparseAdj(to_dev(g.rowptr, dev), to_dev(g.col, dev),
                         None if g.val is None else to_dev(g.val, dev),
                         num_cols=g.K, rows=(b, e))


@pytest.mark.parametrize("N", [16, 64])
def test_banded_range_keeps_the_window_family(sdm, cuda_device, N):
    g = gen.knn_local(20480, 10, 64, seed=11)          # every row has 10 entries: base 10 b
    B = gen.features(g.K, N, seed=11)
    Bd = to_dev(B, cuda_device)
    b, e = 2560, 15360 + 7                             # starts on a 256-row box, ragged end
    adj = _range_adj(sdm, g, cuda_device, b, e)
    adj.set_family("window")
    info = adj.describe(N)
    assert info["row0"] == b and info["M"] == e - b and info["nnz"] == 10 * (e - b)
    assert info["band_w"] == 64 and info["family_name"] == "window", info
    for red in ("sum", "mean"):
        C, A = gpu_reduce(adj, Bd, red)
        compare(g, B, red, C, A, rows=np.arange(b, e), label=f"window range N={N} {red}")
    adj.close()


def test_unaligned_ranges_fall_back_and_stay_exact(sdm, cuda_device):
    g = gen.knn_local(8192, 10, 64, seed=12, weighted=True)
    B = gen.features(g.K, 32, seed=12)
    Bd = to_dev(B, cuda_device)
    for b, e in ((1001, 5003), (1, 2), (0, 8192), (8192, 8192), (4097, 8192)):
        adj = _range_adj(sdm, g, cuda_device, b, e)
        adj.set_family("window")            # not possible: row 1001 starts no tile box
        if b % 128:
            assert adj.describe(32)["family_name"] != "window"
        for red in ("sum", "max"):
            C, A = gpu_reduce(adj, Bd, red)
            compare(g, B, red, C, A, rows=np.arange(b, e), label=f"range [{b},{e}) {red}")
        adj.close()


@pytest.mark.parametrize("parts", [2, 3, 5])
def test_partition_shards_reproduce_the_whole_product(sdm, cuda_device, parts):
    import torch
    g = gen.rmat(scale=14, edge_factor=16, seed=13)    # skewed, heavy rows, empty rows
    B = gen.features(g.K, 64, seed=13)
    Bd = to_dev(B, cuda_device)
    bounds = sdm.spmm_partition_rows(g.rowptr, parts)
    full = make_adj(sdm, g, cuda_device)
    Cf, Af = full.reduce(Bd, "max")
    shards = []
    for q in range(parts):
        adj = _range_adj(sdm, g, cuda_device, bounds[q], bounds[q + 1])
        C, A = adj.reduce(Bd, "max")
        Cs = adj.reduce(Bd, "sum")
        torch.cuda.synchronize()
        compare(g, B, "sum", Cs.cpu().numpy(), None, rows=np.arange(bounds[q], bounds[q + 1]),
                label=f"shard {q} sum")
        shards.append((C, A))
        adj.close()
    C = torch.cat([s[0] for s in shards])
    A = torch.cat([s[1] for s in shards])
    assert torch.equal(C.view(torch.int32), Cf.view(torch.int32)) and torch.equal(A, Af)
    full.close()


def test_range_transpose_and_backward(sdm, cuda_device):
    import oracle
    g = gen.erdos_renyi(3000, 3000, 8, seed=14)
    b, e = 700, 2301
    adj = _range_adj(sdm, g, cuda_device, b, e)
    t = adj.transpose()
    rp = (g.rowptr[b:e + 1] - g.rowptr[b]).astype(np.int32)
    sl = slice(int(g.rowptr[b]), int(g.rowptr[e]))
    rT, cT, vT = oracle.transpose(rp, g.col[sl], g.val[sl], g.K)
    assert np.array_equal(t.rowptr.cpu().numpy(), rT)
    assert np.array_equal(t.col.cpu().numpy(), cT)
    assert np.array_equal(t.val.cpu().numpy().view(np.int32), vT.view(np.int32))
    # d(sum)/dB of the range's rows
    dC = gen.features(e - b, 16, seed=15)
    dB = adj.backward(to_dev(dC, cuda_device), "sum")
    C2, _, T2 = oracle.spmm(rT, cT, vT, dC, "sum", K=e - b)
    err = np.abs(dB.cpu().numpy().astype(np.float64) - C2)
    assert (err <= 1e-5 * T2 + 1e-6).all()
    t.close()
    adj.close()


def test_range_validates_only_its_own_columns(sdm, cuda_device):
    g = gen.erdos_renyi(1024, 1024, 8, seed=16)
    col = g.col.copy()
    col[int(g.rowptr[900])] = 5000                     # out of range, in row 900
    dev = cuda_device
    ok = sdm.SparseAdj(to_dev(g.rowptr, dev), to_dev(col, dev), to_dev(g.val, dev),
                       num_cols=g.K, rows=(0, 512))
    ok.close()
    with pytest.raises(sdm.SpmmError) as err:
        sdm.SparseAdj(to_dev(g.rowptr, dev), to_dev(col, dev), to_dev(g.val, dev),
                      num_cols=g.K, rows=(512, 1024))
    assert err.value.name == "SPMM_ERR_INVALID_INPUT"


def test_block_family_needs_a_range_from_row_zero(sdm, cuda_device):
    g = gen.community(n_comm=8, comm_size=256, seed=17)
    B = gen.features(g.K, 128, seed=17)
    Bd = to_dev(B, cuda_device)
    for b, e in ((0, 1024), (256, 2048)):
        adj = _range_adj(sdm, g, cuda_device, b, e)
        adj.set_family("block")
        fam = adj.describe(128)["family_name"]
        assert fam == ("block" if b == 0 else "warprow"), (b, fam)
        C, A = gpu_reduce(adj, Bd, "sum")
        compare(g, B, "sum", C, A, rows=np.arange(b, e), label=f"block range [{b},{e})")
        adj.close()
