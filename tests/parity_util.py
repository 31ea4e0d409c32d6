"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same inputs, compare.

Tolerance (sum, mean): |gpu - oracle| <= 1e-5 * T + 1e-6 element-wise, with
T = sum_p |a_p * B[col_p, k]| from the oracle. Mean is also held to the
tighter 2e-5 * T / d + 1e-6 (its error is the sum's error divided by d plus
one rounding). Max values and argmax must be bit-identical.
"""
from __future__ import annotations

import numpy as np

import oracle

RTOL = 1e-5
ATOL = 1e-6


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def make_adj(sdm, g, dev, validate=True):
    return sdm.SparseAdj(to_dev(g.rowptr, dev), to_dev(g.col, dev),
                         None if g.val is None else to_dev(g.val, dev),
                         num_cols=g.K, validate=validate)


def gpu_reduce(adj, Bd, reduce, rows=None):
    """Run the engine; return numpy (C, argmax or None), optionally only `rows`."""
    import torch
    res = adj.reduce(Bd, reduce)
    C, A = (res if reduce == "max" else (res, None))
    torch.cuda.synchronize()
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.int64, device=C.device)
        C = C.index_select(0, idx)
        A = None if A is None else A.index_select(0, idx)
    return C.cpu().numpy(), None if A is None else A.cpu().numpy()


def compare(g, B, reduce, C, A, rows=None, label=""):
    Cr, Ar, Tr = oracle.spmm(g.rowptr, g.col, g.val, B, reduce, rows=rows)
    assert C.shape == Cr.shape, (C.shape, Cr.shape)
    if reduce == "max":
        badv = C.view(np.int32) != Cr.view(np.int32)
        assert not badv.any(), f"{label}: {int(badv.sum())} max values differ; first at " \
            f"{np.argwhere(badv)[0]} gpu {C[badv][0]!r} oracle {Cr[badv][0]!r}"
        if A is not None:
            bada = A != Ar
            assert not bada.any(), f"{label}: {int(bada.sum())} argmax differ; first at " \
                f"{np.argwhere(bada)[0]} gpu {A[bada][0]} oracle {Ar[bada][0]}"
        return 0.0
    err = np.abs(C.astype(np.float64) - Cr.astype(np.float64))
    T = Tr.astype(np.float64)
    bound = RTOL * T + ATOL
    bad = err > bound
    assert not bad.any(), f"{label}: {int(bad.sum())} elements outside 1e-5*T+1e-6; worst " \
        f"err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    if reduce == "mean":
        r = np.arange(g.M) if rows is None else np.asarray(rows)
        d = np.diff(g.rowptr.astype(np.int64))[r].astype(np.float64)
        strict = 2 * RTOL * T / np.maximum(d, 1)[:, None] + ATOL
        assert not (err > strict).any(), f"{label}: mean outside 2e-5*T/d+1e-6"
    return float((err / bound).max()) if err.size else 0.0


def sample_rows(g, n, seed=0, t_split=None):
    """Random rows plus the longest rows (and every row above t_split)."""
    rng = np.random.default_rng(seed)
    deg = np.diff(g.rowptr.astype(np.int64))
    pick = [rng.choice(g.M, size=min(n, g.M), replace=False)]
    pick.append(np.argsort(deg)[-64:])
    if t_split is not None:
        pick.append(np.nonzero(deg > t_split)[0])
    pick.append(np.nonzero(deg == 0)[0][:64])
    return np.unique(np.concatenate(pick)).astype(np.int64)
