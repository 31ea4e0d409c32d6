"""Split-precision accuracy of the BLOCK family (tensor cores) on the 64k-row
community graph (256 communities of 256 ids, intra-community probability 0.2
plus 5 outside entries per row), weighted and unweighted, N = 128 and 512.

RA-SpMM's blocked tensor-core families ("kernel composition") take FP16/TF32
operands directly. For each element the error is measured against the oracle
in units of the sum tolerance, err / (1e-5 * T + 1e-6):

* split TF32 (the kernel: x = hi + lo, hi * hi + hi * lo + lo * hi) must stay
  below 1 everywhere;
* plain TF32 (one rounding of each operand, products exact, sums exact) is
  evaluated on the host from the same operands for comparison; its worst
  element is expected above 1, i.e. outside the tolerance.
"""
import numpy as np
import pytest

import gen
import oracle
from parity_util import ATOL, RTOL, make_adj, to_dev

pytestmark = pytest.mark.gpu

_g = {}


def community(weighted):
    if "w" not in _g:
        _g["w"] = gen.config(4)
    g = _g["w"]
    return g if weighted else gen.Graph(g.name + "_u", g.M, g.K, g.rowptr, g.col, None)


def tf32(x):
    """Round to nearest TF32 (10 explicit mantissa bits), ties away from zero."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def plain_tf32_product(g, B):
    """Entries inside their row's 256-column diagonal block with TF32 operands
    (the tensor-core part), the others exact; all sums in fp64."""
    import scipy.sparse as sp
    rows = np.repeat(np.arange(g.M), np.diff(g.rowptr.astype(np.int64)))
    a = np.ones(g.nnz, np.float32) if g.val is None else g.val
    in_blk = (g.col // 256) == (rows // 256)
    a_blk = np.where(in_blk, tf32(a), 0.0).astype(np.float64)
    a_off = np.where(in_blk, 0.0, a).astype(np.float64)
    Ab = sp.csr_matrix((a_blk, g.col, g.rowptr), shape=(g.M, g.K))
    Ao = sp.csr_matrix((a_off, g.col, g.rowptr), shape=(g.M, g.K))
    return Ab @ tf32(B).astype(np.float64) + Ao @ B.astype(np.float64)


@pytest.mark.parametrize("weighted", [True, False])
@pytest.mark.parametrize("N", [128, 512])
def test_split_tf32_within_tolerance_plain_tf32_not(cuda_device, weighted, N):
    import torch
    import sparse_dense_matrix_gb300 as sdm
    g = community(weighted)
    B = gen.features(g.K, N, seed=0)
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family("block")
    assert adj.describe(N, "sum")["family_name"] == "block"
    C = adj.reduce(to_dev(B, cuda_device), "sum")
    torch.cuda.synchronize()
    C = C.cpu().numpy().astype(np.float64)
    Cr, _, T = oracle.spmm(g.rowptr, g.col, g.val, B, "sum")
    bound = RTOL * T.astype(np.float64) + ATOL
    split = float((np.abs(C - Cr) / bound).max())
    plain = float((np.abs(plain_tf32_product(g, B) - Cr) / bound).max())
    print(f"community 64k {'weighted' if weighted else 'unweighted'} N={N}: "
          f"max err / tolerance: split TF32 {split:.3g}, plain TF32 {plain:.3g}")
    assert split < 1.0
    assert plain > 1.0
    adj.close()
