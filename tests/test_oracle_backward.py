"""Pins of the oracle's backward definitions (CPU):

* the transpose against a stable sort of the entries by column (numpy);
* the sum and mean backward, composed as a product with the transpose, against
  torch autograd of the dense fp64 forward;
* the max-pool backward against torch autograd of a per-entry maximum (each
  row's stored entries padded to the longest row, duplicated pairs included,
  so that autograd routes the gradient through the one entry that won), and
  against hand-worked duplicated pairs whose winner is fixed by the sign of
  B (largest product) or by a tie (first copy).
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


def per_entry_max_grad(g, B0, dC):
    """Autograd of C[i, k] = max over the stored entries p of row i of
    a_p * B[col_p, k] (rows padded to the longest with -inf; empty rows give
    no gradient). Duplicated pairs stay separate entries, so the gradient
    reaches B only through the entry torch.max picked."""
    deg = g.degrees()
    dmax = max(1, int(deg.max()))
    M, N = dC.shape
    idx = np.zeros((g.M, dmax), np.int64)
    a = np.zeros((g.M, dmax), np.float64)
    live = np.zeros((g.M, dmax), bool)
    for i in range(g.M):
        p0, p1 = g.rowptr[i], g.rowptr[i + 1]
        idx[i, :p1 - p0] = g.col[p0:p1]
        a[i, :p1 - p0] = 1.0 if g.val is None else g.val[p0:p1]
        live[i, :p1 - p0] = True
    B = torch.tensor(B0.astype(np.float64), requires_grad=True)
    prod = torch.from_numpy(a)[:, :, None] * B[torch.from_numpy(idx)]       # [M, dmax, N]
    prod = torch.where(torch.from_numpy(live)[:, :, None], prod, torch.full_like(prod, -np.inf))
    Cd = prod.max(dim=1).values
    has = torch.from_numpy(deg > 0)
    (torch.where(has[:, None], Cd, torch.zeros_like(Cd)) *
     torch.from_numpy(dC.astype(np.float64))).sum().backward()
    return B.grad.numpy()


@pytest.mark.parametrize("seed", [5, 6, 7])
@pytest.mark.parametrize("weighted", [True, False])
def test_maxpool_backward_matches_autograd(seed, weighted):
    # duplicated pairs: weighted copies carry different values (one of them
    # wins); unweighted copies are equal, and any one of them gives dC once
    g = random_graph(seed, dup=True, weighted=weighted)
    assert any(len(set(g.col[g.rowptr[i]:g.rowptr[i + 1]])) < g.rowptr[i + 1] - g.rowptr[i]
               for i in range(g.M)), "the pin needs duplicated pairs"
    N = 5
    rng = np.random.default_rng(seed)
    B0 = rng.standard_normal((g.K, N)).astype(np.float32)
    dC = rng.standard_normal((g.M, N)).astype(np.float32)
    C, A, _ = oracle.spmm(g.rowptr, g.col, g.val, B0, "max")
    want = per_entry_max_grad(g, B0, dC)
    got = oracle.maxpool_backward(g.rowptr, g.col, g.val, A, dC, g.K, B0)
    assert np.allclose(got, want, rtol=1e-6, atol=1e-6)


def test_maxpool_backward_duplicate_winner_by_hand():
    """One row holding column 0 three times (weights 2, 3, 2) and column 1 once
    (weight 1); dC = 1. Worked out by hand from the definition:
      k = 0, B[0] = +1: products 2, 3, 2 and 1 -> the copy of weight 3 wins, dB[0] = 3;
      k = 1, B[0] = -1, B[1] = -5: products -2, -3, -2 and -5 -> column 0, and
             the first copy of weight 2 wins the tie with the third, dB[0] = 2;
      k = 2, B[0] = 0, B[1] = -1: products 0, 0, 0 and -1 -> column 0, a tie of
             all three copies, the first (weight 2) wins, dB[0] = 2.
    Counting every copy of the winning pair (the rule this replaces) would give
    7, 7 and 7."""
    g = gen.from_rows("dup", 1, 2, [[0, 0, 1, 0]], [[2.0, 3.0, 1.0, 2.0]])
    B0 = np.array([[1.0, -1.0, 0.0], [1.0, -5.0, -1.0]], np.float32)
    dC = np.ones((1, 3), np.float32)
    C, A, _ = oracle.spmm(g.rowptr, g.col, g.val, B0, "max")
    assert A.tolist() == [[0, 0, 0]]
    assert C.tolist() == [[3.0, -2.0, 0.0]]
    dB = oracle.maxpool_backward(g.rowptr, g.col, g.val, A, dC, g.K, B0)
    assert dB.tolist() == [[3.0, 2.0, 2.0], [0.0, 0.0, 0.0]]
    # unweighted: the three copies of column 0 are equal and the gradient
    # passes once (k = 0: B[1] = 2 beats B[0] = 1, column 1 wins)
    gu = gen.from_rows("dupu", 1, 2, [[0, 0, 1, 0]], None)
    Bu = np.array([[1.0, -1.0, 0.0], [2.0, -5.0, -1.0]], np.float32)
    Cu, Au, _ = oracle.spmm(gu.rowptr, gu.col, None, Bu, "max")
    dBu = oracle.maxpool_backward(gu.rowptr, gu.col, None, Au, dC, gu.K)
    assert Au.tolist() == [[1, 0, 0]]
    assert dBu.tolist() == [[0.0, 1.0, 1.0], [1.0, 0.0, 0.0]]
