"""Pins of the oracle's backward definitions (CPU):

* the transpose against a stable sort of the entries by column (numpy);
* the sum and mean backward, composed as a product with the transpose, against
  torch autograd of the dense fp64 forward;
* the max-pool backward against torch autograd of a dense masked maximum
  (continuous values, no ties, no duplicate pairs).
"""
import numpy as np
import pytest

import gen
import oracle

torch = pytest.importorskip("torch")


def random_graph(seed, M=37, K=29, max_deg=9, dup=True, weighted=True):
    rng = np.random.default_rng(seed)
    rows, vals = [], []
    for i in range(M):
        d = 0 if rng.random() < 0.15 else int(rng.integers(1, max_deg + 1))
        c = rng.choice(K, size=min(d, K), replace=False).tolist()
        if dup and len(c) >= 2 and rng.random() < 0.4:
            c[-1] = c[0]
        rng.shuffle(c)
        rows.append(c)
        vals.append(rng.standard_normal(len(c)).astype(np.float32).tolist())
    return gen.from_rows("g", M, K, rows, vals if weighted else None)


def dense(g, dtype=torch.float64):
    A = torch.zeros((g.M, g.K), dtype=dtype)
    deg = g.degrees()
    r = torch.from_numpy(np.repeat(np.arange(g.M), deg))
    c = torch.from_numpy(g.col.astype(np.int64))
    v = torch.ones(g.nnz, dtype=dtype) if g.val is None else torch.from_numpy(g.val).to(dtype)
    A.index_put_((r, c), v, accumulate=True)
    return A


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("weighted", [True, False])
def test_transpose_is_a_stable_sort_by_column(seed, weighted):
    g = random_graph(seed, weighted=weighted)
    rT, cT, vT = oracle.transpose(g.rowptr, g.col, g.val, g.K)
    rows = np.repeat(np.arange(g.M), g.degrees())
    order = np.argsort(g.col, kind="stable")
    assert np.array_equal(cT, rows[order])
    assert np.array_equal(rT, np.concatenate([[0], np.cumsum(np.bincount(g.col, minlength=g.K))]))
    if weighted:
        assert np.array_equal(vT, g.val[order])
    else:
        assert vT is None


@pytest.mark.parametrize("seed", [3, 4])
def test_sum_and_mean_backward_match_autograd(seed):
    g = random_graph(seed)
    N = 6
    rng = np.random.default_rng(seed)
    B0 = rng.standard_normal((g.K, N))
    dC = rng.standard_normal((g.M, N)).astype(np.float32)
    A = dense(g)
    deg = torch.from_numpy(g.degrees().astype(np.float64)).clamp(min=1)[:, None]
    for red, scale in (("sum", False), ("mean", True)):
        B = torch.tensor(B0, requires_grad=True)
        C = A @ B
        if red == "mean":
            C = C / deg
        (C * torch.from_numpy(dC.astype(np.float64))).sum().backward()
        want = B.grad.numpy()
        rT, cT, vT = oracle.transpose(g.rowptr, g.col, g.val, g.K, scale_mean=scale)
        got, _, T = oracle.spmm(rT, cT, vT, dC, "sum")
        assert np.all(np.abs(got - want) <= 2.0 ** -22 * np.abs(want) + 1e-6 * (T + 1)), red


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_maxpool_backward_matches_autograd(seed):
    g = random_graph(seed, dup=False)
    N = 5
    rng = np.random.default_rng(seed)
    B0 = rng.standard_normal((g.K, N)).astype(np.float32)
    dC = rng.standard_normal((g.M, N)).astype(np.float32)
    C, A, _ = oracle.spmm(g.rowptr, g.col, g.val, B0, "max")
    # dense masked maximum over stored entries; rows without entries have no gradient
    Ad = dense(g)
    mask = torch.zeros((g.M, g.K), dtype=torch.bool)
    deg = g.degrees()
    mask[torch.from_numpy(np.repeat(np.arange(g.M), deg)), torch.from_numpy(g.col.astype(np.int64))] = True
    B = torch.tensor(B0.astype(np.float64), requires_grad=True)
    prod = Ad[:, :, None] * B[None, :, :]                         # [M, K, N]
    prod = torch.where(mask[:, :, None], prod, torch.full_like(prod, -np.inf))
    has = torch.from_numpy(deg > 0)
    Cd = prod.max(dim=1).values
    (torch.where(has[:, None], Cd, torch.zeros_like(Cd)) *
     torch.from_numpy(dC.astype(np.float64))).sum().backward()
    want = B.grad.numpy()
    got = oracle.maxpool_backward(g.rowptr, g.col, g.val, A, dC, g.K)
    assert np.allclose(got, want, rtol=1e-6, atol=1e-6)
