"""The five measured workloads at full size, in the launch configuration the
benchmark times (router's choice, default split threshold).

Where the oracle finishes in seconds every output element is compared;
otherwise a sample of rows (random rows, the longest rows, every split row,
some empty rows) is computed by the oracle one by one and compared.
"""
import numpy as np
import pytest

import gen
from parity_util import compare, gpu_reduce, make_adj, sample_rows, to_dev

pytestmark = pytest.mark.gpu

_graphs = {}


def graph(cid):
    if cid not in _graphs:
        _graphs.clear()                        # hold one full-size graph at a time
        _graphs[cid] = gen.config(cid)
    return _graphs[cid]


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


# (config, N, reduce, full comparison?)
CASES = [(1, 32, r, True) for r in ("sum", "mean", "max")]
CASES += [(2, n, r, True) for n in (16, 64) for r in ("sum", "mean")]
CASES += [(3, 64, r, True) for r in ("sum", "max")]
CASES += [(3, n, r, False) for n in (128, 256) for r in ("sum", "max")]
CASES += [(4, n, "sum", True) for n in (128, 512)]
CASES += [(5, 16, r, True) for r in ("sum", "mean", "max")]
CASES += [(5, n, r, False) for n in (32, 64, 128, 256) for r in ("sum", "mean", "max")]


@pytest.mark.parametrize("cid,N,red,full", CASES,
                         ids=[f"c{c}-N{n}-{r}" for c, n, r, _ in CASES])
def test_workload(sdm, cuda_device, cid, N, red, full):
    import torch
    g = graph(cid)
    adj = make_adj(sdm, g, cuda_device)
    info = adj.describe(N, red)
    B = gen.features(g.K, N, seed=0)
    Bd = to_dev(B, cuda_device)
    rows = None if full else sample_rows(g, 20000, seed=cid * 1000 + N, t_split=info["t_split"])
    C, A = gpu_reduce(adj, Bd, red, rows=rows)
    compare(g, B, red, C, A, rows=rows, label=f"config {cid} N={N} {red} ({info['family_name']})")
    del Bd
    adj.close()
    torch.cuda.empty_cache()
