"""spmm_run_noalloc: the product without a plan and without device allocation,
for callers whose device memory belongs to another allocator or who must not
allocate after start-up. Checked element by element against the oracle (the
same tolerance and bit-exact max/argmax as every other parity test) on
consecutive calls, which share the library's one static scratch array, and
cross-checked against the planned entry point (spmm_run through SparseAdj).
After a first call, further calls must leave the device's free memory
unchanged. This file is collected last on purpose."""
import numpy as np
import pytest

import gen
from parity_util import ATOL, RTOL, compare, make_adj, to_dev

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


def test_noalloc_matches_oracle_on_consecutive_calls(sdm, cuda_device):
    import oracle
    g = gen.rmat(scale=13, edge_factor=16, seed=4)
    deg = g.degrees()
    t_split = sdm.spmm_default_t_split(g.M, g.nnz, 152)
    assert (deg > t_split).any()                  # the split path and its scratch are used
    adj = make_adj(sdm, g, cuda_device)
    n0 = sdm.spmm_launch_count()
    for N, red in ((32, "sum"), (64, "max"), (32, "mean"), (64, "max")):
        B = gen.features(g.K, N, seed=N + 11)
        Bd = to_dev(B, cuda_device)
        C1, A1 = _noalloc(sdm, g, cuda_device, Bd, red)
        compare(g, B, red, C1, A1, label=f"noalloc N={N} {red}")
        # the planned entry point on the same input: max bit for bit, the sums
        # both within the oracle's tolerance, hence within twice it of each other
        C0, A0 = _planned(sdm, adj, Bd, red)
        if red == "max":
            assert np.array_equal(C1.view(np.int32), C0.view(np.int32))
            assert np.array_equal(A1, A0)
        else:
            _, _, T = oracle.spmm(g.rowptr, g.col, g.val, B, red)
            err = np.abs(C1.astype(np.float64) - C0.astype(np.float64))
            assert np.all(err <= 2 * (RTOL * T.astype(np.float64) + ATOL)), red
    assert sdm.spmm_launch_count() > n0
    adj.close()


def test_noalloc_allocates_nothing(sdm, cuda_device):
    """Once the library is loaded and the array's address looked up (the first
    call), calls change neither the device's free memory nor torch's."""
    import torch
    g = gen.chung_lu(1 << 14, 2.1, 25.0, 2000.0, seed=3)
    N = 64
    B = gen.features(g.K, N, seed=5)
    rp, cl, vl = to_dev(g.rowptr, cuda_device), to_dev(g.col, cuda_device), to_dev(g.val, cuda_device)
    Bd = to_dev(B, cuda_device)
    C = torch.empty((g.M, N), dtype=torch.float32, device=cuda_device)
    A = torch.empty((g.M, N), dtype=torch.int32, device=cuda_device)

    def call(red):
        sdm.spmm_run_noalloc(rp.data_ptr(), cl.data_ptr(), vl.data_ptr(), Bd.data_ptr(), g.M,
                             g.K, N, sdm.REDUCE[red], C.data_ptr(),
                             A.data_ptr() if red == "max" else None)

    call("sum")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda_device)
    torch0 = torch.cuda.memory_reserved(cuda_device)
    for red in ("sum", "max", "mean", "sum"):
        call(red)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda_device)
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_reserved(cuda_device) == torch0
    compare(g, B, "sum", C.cpu().numpy(), None, label="noalloc after the memory check")


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
    B = gen.features(K, 8, seed=1)
    Bd = to_dev(B, cuda_device)
    C1, _ = _noalloc(sdm, g, cuda_device, Bd, "sum")
    compare(g, B, "sum", C1, None, label="noalloc after a refusal")
