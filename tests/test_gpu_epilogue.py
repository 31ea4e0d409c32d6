"""Fused epilogue C = act(R + bias) (spmm_run_ex) on the GPU vs the oracle.

Every family writes C in its own store path, so each is pinned here: sum and
mean within 1e-5 * (T + |bias|) + 1e-6 (the bias adds one fp32 rounding of a
value of at most T + |bias|); max values and argmax bit-identical (both sides
add the bias to the same fp32 maximum with one rounding).
"""
import numpy as np
import pytest

import gen
import oracle
from parity_util import ATOL, RTOL, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


_cache = {}


def graph(name):
    if name not in _cache:
        _cache[name] = {
            "er": lambda: gen.erdos_renyi(3000, 2500, 8, seed=1),
            "knn": lambda: gen.knn_local(20000, 10, 512, seed=1),
            "rmat": lambda: gen.rmat(scale=13, edge_factor=16, seed=1),
        }[name]()
    return _cache[name]


def check(sdm, dev, g, N, red, bias, act, family="auto", t_split=0):
    import torch
    B = gen.features(g.K, N, seed=N + 3)
    adj = make_adj(sdm, g, dev)
    adj.set_family(family, t_split)
    fam = adj.describe(N, red)["family_name"]
    bd = None if bias is None else to_dev(bias, dev)
    res = adj.reduce(to_dev(B, dev), red, bias=bd, activation=act)
    C, A = res if red == "max" else (res, None)
    torch.cuda.synchronize()
    C = C.cpu().numpy()
    Cr, Ar, Tr = oracle.spmm(g.rowptr, g.col, g.val, B, red, bias=bias, act=act or "none")
    label = f"{g.name} {fam} N={N} {red} bias={bias is not None} act={act}"
    if red == "max":
        assert np.array_equal(C.view(np.int32), Cr.view(np.int32)), label
        assert np.array_equal(A.cpu().numpy(), Ar), label
    else:
        T = Tr.astype(np.float64) + (0 if bias is None else np.abs(bias.astype(np.float64)))
        err = np.abs(C.astype(np.float64) - Cr.astype(np.float64))
        assert not (err > RTOL * T + ATOL).any(), label
    adj.close()
    return fam


@pytest.mark.parametrize("family,name,t_split", [
    ("rowgroup", "er", 0), ("warprow", "rmat", 0), ("warprow", "rmat", 40),
    ("window", "knn", 0), ("coltile", "er", 0)])
@pytest.mark.parametrize("N", [4, 33, 64, 160])
@pytest.mark.parametrize("red", ["sum", "mean", "max"])
def test_epilogue_every_family(sdm, cuda_device, family, name, t_split, N, red):
    g = graph(name)
    bias = gen.features(1, N, seed=N)[0]
    fam = check(sdm, cuda_device, g, N, red, bias, "relu", family, t_split)
    if family == "window" and N % 4 == 0:
        assert fam == "window"


@pytest.mark.parametrize("bias_on,act", [(True, None), (False, "relu"), (False, None)])
def test_epilogue_parts(sdm, cuda_device, bias_on, act):
    g = graph("er")
    N = 16
    bias = gen.features(1, N, seed=1)[0] if bias_on else None
    for red in ("sum", "mean", "max"):
        check(sdm, cuda_device, g, N, red, bias, act)


def test_epilogue_arguments(sdm, cuda_device):
    import torch
    g = graph("er")
    adj = make_adj(sdm, g, cuda_device)
    B = to_dev(gen.features(g.K, 8, seed=2), cuda_device)
    with pytest.raises(ValueError):
        adj.reduce(B, "sum", activation="gelu")
    with pytest.raises(ValueError):
        adj.reduce(B, "sum", bias=torch.zeros(7, device=cuda_device))
    C = torch.empty(g.M, 8, device=cuda_device)
    with pytest.raises(sdm.SpmmError):
        sdm.spmm_run_ex(adj.plan, adj.col.data_ptr(), adj.val.data_ptr(), B.data_ptr(), 8, 0,
                        None, 5, C.data_ptr())
    adj.close()
