"""Outputs past 2^31 elements: C and argmax of 2,100,000 rows x 1,024 columns
(2.15e9 elements each, 8.6 GB), so every row index above 2,097,151 needs 64-bit
output offsets. Each family that takes this width is held to the oracle on
the rows around the 2^31 boundary, the rows past it, the long rows placed at
the end (the split-row path) and a seeded sample of the rest."""
import numpy as np
import pytest

import gen
from parity_util import compare, gpu_reduce, make_adj, to_dev

pytestmark = pytest.mark.gpu

M, K, N = 2_100_000, 1_000, 1_024
EDGE = (1 << 31) // N                  # first row whose output offset needs 64 bits


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


@pytest.fixture(scope="module")
def big_graph():
    """Two random entries per row; the last 8 rows hold 3,000 entries each,
    more than the split threshold."""
    rng = np.random.default_rng(11)
    deg = np.full(M, 2, dtype=np.int64)
    deg[-8:] = 3000
    rowptr = np.zeros(M + 1, dtype=np.int32)
    rowptr[1:] = np.cumsum(deg)
    nnz = int(rowptr[-1])
    col = rng.integers(0, K, size=nnz).astype(np.int32)
    val = rng.random(nnz, dtype=np.float32)
    return gen.Graph("wide_out", M, K, rowptr, col, val)


@pytest.mark.parametrize("family", ["auto", "segment", "stream", "gather", "coltile"])
def test_outputs_past_2_31_elements(sdm, cuda_device, big_graph, family):
    import torch
    free, _ = torch.cuda.mem_get_info(cuda_device)
    if free < 40 << 30:
        pytest.skip(f"needs 40 GB of free device memory, {free >> 30} GB free")
    g = big_graph
    B = gen.features(K, N, seed=12)
    Bd = to_dev(B, cuda_device)
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([np.arange(EDGE - 64, EDGE + 64), np.arange(M - 3000, M),
                                     rng.integers(0, M, 2000)]))
    adj = make_adj(sdm, g, cuda_device)
    adj.set_family(family)
    for red in ("sum", "max"):
        info = adj.describe(N, red)
        if family != "auto":
            assert info["family_name"] == family, info
        C, A = gpu_reduce(adj, Bd, red, rows=rows)
        compare(g, B, red, C, A, rows=rows, label=f"{info['family_name']} {red} M={M} N={N}")
        torch.cuda.empty_cache()
    adj.close()
