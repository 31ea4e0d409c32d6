"""spmm_run_noalloc: the product without a plan and without device allocation,
for callers whose device memory belongs to another allocator or who must not
allocate after start-up. Checked against the planned entry point (spmm_run
through SparseAdj) on consecutive calls, which share the library's one static
scratch array. This file is collected last on purpose."""
import numpy as np
import pytest

import gen
from parity_util import ATOL, RTOL, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


def _noalloc(sdm, g, dev, Bd, red):
    import torch
    N = Bd.shape[1]
    rp, cl = to_dev(g.rowptr, dev), to_dev(g.col, dev)
    vl = None if g.val is None else to_dev(g.val, dev)
    C = torch.full((g.M, N), float("nan"), dtype=torch.float32, device=dev)
    A = torch.full((g.M, N), -7, dtype=torch.int32, device=dev) if red == "max" else None
    sdm.spmm_run_noalloc(rp.data_ptr(), cl.data_ptr(), None if vl is None else vl.data_ptr(),
                         Bd.data_ptr(), g.M, g.K, N, sdm.REDUCE[red], C.data_ptr(),
                         None if A is None else A.data_ptr())
    torch.cuda.synchronize()
    return C.cpu().numpy(), None if A is None else A.cpu().numpy()


def _planned(sdm, adj, Bd, red):
    import torch
    r = adj.reduce(Bd, red)
    torch.cuda.synchronize()
    if red == "max":
        return r[0].cpu().numpy(), r[1].cpu().numpy()
    return r.cpu().numpy(), None


def test_noalloc_matches_planned_entry_point_on_consecutive_calls(sdm, cuda_device):
    import oracle
    g = gen.rmat(scale=13, edge_factor=16, seed=4)
    deg = g.degrees()
    t_split = sdm.spmm_default_t_split(g.M, g.nnz, 152)
    assert (deg > t_split).any()                  # the split path and its scratch are used
    adj = make_adj(sdm, g, cuda_device)
    n0 = sdm.spmm_launch_count()
    for N, red in ((32, "sum"), (64, "max"), (32, "mean")):
        B = gen.features(g.K, N, seed=N + 11)
        Bd = to_dev(B, cuda_device)
        C1, A1 = _noalloc(sdm, g, cuda_device, Bd, red)
        C0, A0 = _planned(sdm, adj, Bd, red)
        if red == "max":
            assert np.array_equal(C1.view(np.int32), C0.view(np.int32))
            assert np.array_equal(A1, A0)
        else:
            _, _, T = oracle.spmm(g.rowptr, g.col, g.val, B, red)
            err = np.abs(C1.astype(np.float64) - C0.astype(np.float64))
            assert np.all(err <= 2 * (RTOL * T.astype(np.float64) + ATOL)), red
    assert sdm.spmm_launch_count() > n0


def test_noalloc_rejects_inputs_beyond_its_scratch(sdm, cuda_device):
    import torch
    # one row of 200,000 entries -> 1,563 chunks; at N = 16,384 the partials
    # (about 102 MB) exceed the static array, so the call must refuse
    rng = np.random.default_rng(2)
    K, N = 64, 16384
    g = gen.from_rows("long", 1, K, [rng.integers(0, K, size=200_000).tolist()])
    Bd = torch.zeros((K, N), dtype=torch.float32, device=cuda_device)
    with pytest.raises(sdm.SpmmError) as e:
        _noalloc(sdm, g, cuda_device, Bd, "sum")
    assert e.value.status == 5                    # SPMM_ERR_UNSUPPORTED
    # a size that fits still works after the refusal
    import oracle
    B = gen.features(K, 8, seed=1)
    Bd = to_dev(B, cuda_device)
    C1, _ = _noalloc(sdm, g, cuda_device, Bd, "sum")
    C0, _ = _planned(sdm, make_adj(sdm, g, cuda_device), Bd, "sum")
    _, _, T = oracle.spmm(g.rowptr, g.col, g.val, B, "sum")
    err = np.abs(C1.astype(np.float64) - C0.astype(np.float64))
    assert np.all(err <= 2 * (RTOL * T.astype(np.float64) + ATOL))
