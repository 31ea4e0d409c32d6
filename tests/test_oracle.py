"""Pins of the CPU oracle to things other than itself.

* a hand-worked fixture (tests/golden/hand_4x3.json) with duplicates, an empty
  row, unsorted columns and signed-zero ties;
* dense fp64 products from scipy.sparse / numpy on tiny random inputs
  (duplicates summed by scipy's CSR product);
* closed forms: identity and ring graphs, B = ones (weighted row sums),
  constant B (argmax = smallest column), row-normalised values (row sums 1);
* edge semantics of the graph-spmm model card ("Correctness"): unweighted ==
  all-ones values, empty rows, duplicates summed, tie to the smallest column;
* the degree descriptors against closed forms.

test_planted_mistake_is_caught builds the oracle with one planted mistake at a
time (a dropped term, a wrong index, a transposed operand, a reversed tie rule,
a wrong mean divisor) and checks that at least one pin rejects each.
"""
import json
import os

import numpy as np
import pytest
import scipy.sparse as sp

import gen
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def random_csr(rng, M, K, max_deg, dup=True, sort=False, empty_frac=0.2, weighted=True):
    rows = []
    vals = []
    for _ in range(M):
        d = 0 if rng.random() < empty_frac else int(rng.integers(1, max_deg + 1))
        c = list(rng.integers(0, K, size=d))
        if dup and d >= 2 and rng.random() < 0.5:
            c[-1] = c[0]
        if sort:
            c.sort()
        rows.append(c)
        vals.append(list(rng.standard_normal(d).astype(np.float32)))
    g = gen.from_rows("rand", M, K, rows, vals if weighted else None)
    return g


def dense_fp64(g, absolute=False):
    """A as a sparse fp64 matrix; scipy sums duplicate (row, col) entries."""
    val = np.ones(g.nnz) if g.val is None else g.val.astype(np.float64)
    if absolute:
        val = np.abs(val)
    A = sp.csr_matrix((val, g.col.astype(np.int64), g.rowptr.astype(np.int64)), shape=(g.M, g.K))
    return A


def pin_golden_hand_worked(o):
    fx = json.load(open(os.path.join(HERE, "golden", "hand_4x3.json")))
    rowptr = np.array(fx["rowptr"], np.int32)
    col = np.array(fx["col"], np.int32)
    val = np.array(fx["val"], np.float32)
    B = np.array(fx["B"], np.float32)
    C, _, _ = o.spmm(rowptr, col, val, B, "sum")
    assert np.array_equal(C, np.array(fx["sum"], np.float32))
    C, _, _ = o.spmm(rowptr, col, val, B, "mean")
    want = (np.array(fx["mean_num"], np.float64) / np.array(fx["mean_den"], np.float64)[:, None])
    assert np.array_equal(C, want.astype(np.float32))
    C, A, _ = o.spmm(rowptr, col, val, B, "max")
    assert np.array_equal(C, np.array(fx["max"], np.float32))
    assert np.array_equal(np.signbit(C), np.array(fx["max_signbit"]))
    assert np.array_equal(A, np.array(fx["argmax"], np.int32))


def pin_sum_mean_match_dense_fp64(o):
    for N in (1, 3, 17, 32):
        for seed in (0, 1, 2):
            _dense_case(o, N, seed)


def _dense_case(o, N, seed):
    rng = np.random.default_rng(100 + seed)
    M, K = int(rng.integers(1, 65)), int(rng.integers(1, 65))
    g = random_csr(rng, M, K, max_deg=12)
    B = rng.standard_normal((K, N)).astype(np.float32)
    ref = dense_fp64(g) @ B.astype(np.float64)
    C, _, T = o.spmm(g.rowptr, g.col, g.val, B, "sum")
    # only the last fp32 rounding (and fp64 order noise far below it) may differ
    tol = np.abs(ref) * 2.0 ** -24 + 1e-12 * T.astype(np.float64) + 1e-300
    assert np.all(np.abs(C.astype(np.float64) - ref) <= tol)
    absref = dense_fp64(g, absolute=True) @ np.abs(B.astype(np.float64))
    assert np.allclose(T, absref, rtol=1e-6, atol=0)  # T = sum |a b| over stored entries
    deg = g.degrees()
    Cm, _, _ = o.spmm(g.rowptr, g.col, g.val, B, "mean")
    refm = np.where(deg[:, None] > 0, ref / np.maximum(deg, 1)[:, None], 0.0)
    tolm = np.abs(refm) * 2.0 ** -24 + 1e-12 * T.astype(np.float64) + 1e-300
    assert np.all(np.abs(Cm.astype(np.float64) - refm) <= tolm)


def pin_max_matches_set_maximum(o):
    for N in (1, 4, 9):
        for seed in (0, 1, 2, 3):
            _max_case(o, N, seed)


def _max_case(o, N, seed):
    """Max as a set maximum over fp32 products (numpy float32 multiply is correctly
    rounded); argmax = smallest column among the entries attaining it."""
    rng = np.random.default_rng(200 + seed)
    M, K = 40, 30
    g = random_csr(rng, M, K, max_deg=9)
    # a coarse value grid makes exact ties frequent
    B = (rng.integers(-3, 4, size=(K, N))).astype(np.float32)
    g.val = rng.integers(-2, 3, size=g.nnz).astype(np.float32)
    C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, "max")
    for i in range(M):
        p0, p1 = g.rowptr[i], g.rowptr[i + 1]
        if p0 == p1:
            assert np.all(C[i] == 0) and np.all(A[i] == -1)
            continue
        P = g.val[p0:p1, None] * B[g.col[p0:p1]]          # float32 products [d, N]
        mx = P.max(axis=0)
        assert np.array_equal(C[i], mx)
        cols = np.where(P == mx[None, :], g.col[p0:p1, None], np.iinfo(np.int32).max)
        assert np.array_equal(A[i], cols.min(axis=0))


def pin_identity_graph(o):
    M, N = 50, 7
    g = gen.from_rows("eye", M, M, [[i] for i in range(M)])
    B = gen.features(M, N, seed=3)
    for red in ("sum", "mean", "max"):
        C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, red)
        assert np.array_equal(C, B)
        if red == "max":
            assert np.array_equal(A, np.repeat(np.arange(M, dtype=np.int32)[:, None], N, 1))


def pin_ring_graph(o):
    M, N = 37, 5
    rows = [[(i - 1) % M, (i + 1) % M] for i in range(M)]
    g = gen.from_rows("ring", M, M, rows)
    B = gen.features(M, N, seed=4)
    B64 = B.astype(np.float64)
    prev = np.roll(B64, 1, axis=0)     # B[i-1]
    nxt = np.roll(B64, -1, axis=0)     # B[i+1]
    C, _, _ = o.spmm(g.rowptr, g.col, None, B, "sum")
    assert np.array_equal(C, (prev + nxt).astype(np.float32))  # exact fp64 sum, rounded once
    C, _, _ = o.spmm(g.rowptr, g.col, None, B, "mean")
    assert np.array_equal(C, ((prev + nxt) / 2).astype(np.float32))
    C, A, _ = o.spmm(g.rowptr, g.col, None, B, "max")
    assert np.array_equal(C, np.maximum(prev, nxt).astype(np.float32))
    ci = np.array([r for r in rows], dtype=np.int32)       # [M, 2] columns (i-1, i+1)
    pick_prev = (prev > nxt) | ((prev == nxt) & (ci[:, 0:1] < ci[:, 1:2]))
    want = np.where(pick_prev, ci[:, 0:1], ci[:, 1:2])
    assert np.array_equal(A, want)


def pin_ones_gives_weighted_row_sums(o):
    g = gen.erdos_renyi(300, 200, 6, seed=5)
    B = np.ones((g.K, 3), np.float32)
    rs = np.add.reduceat(np.concatenate([g.val.astype(np.float64), [0.0]]),
                         g.rowptr[:-1].astype(np.int64))[: g.M]
    C, _, _ = o.spmm(g.rowptr, g.col, g.val, B, "sum")
    assert np.array_equal(C, np.repeat(rs.astype(np.float32)[:, None], 3, 1))
    C, _, _ = o.spmm(g.rowptr, g.col, g.val, B, "mean")
    assert np.array_equal(C, np.repeat((rs / 6).astype(np.float32)[:, None], 3, 1))
    C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, "max")
    for i in range(g.M):
        seg = g.val[g.rowptr[i]:g.rowptr[i + 1]]
        cols = g.col[g.rowptr[i]:g.rowptr[i + 1]]
        assert np.all(C[i] == seg.max())
        assert np.all(A[i] == cols[seg == seg.max()].min())


def pin_row_normalised_rows_sum_to_one(o):
    g = gen.rmat(scale=10, edge_factor=8, seed=1)
    B = np.ones((g.K, 2), np.float32)
    C, _, T = o.spmm(g.rowptr, g.col, g.val, B, "sum")
    deg = g.degrees()
    assert np.all(C[deg == 0] == 0)
    assert np.all(np.abs(C[deg > 0] - 1.0) <= 1e-6 * deg[deg > 0, None])


def pin_constant_B_argmax_is_smallest_column_even_unsorted(o):
    rows = [[9, 4, 7, 4], [3], [], [8, 1, 1]]
    g = gen.from_rows("u", 4, 10, rows)
    B = np.full((10, 3), 2.5, np.float32)
    C, A, _ = o.spmm(g.rowptr, g.col, None, B, "max")
    assert np.array_equal(A[:, 0], [4, 3, -1, 1])
    assert np.array_equal(C[:, 0], [2.5, 2.5, 0.0, 2.5])


def pin_unweighted_equals_all_ones_and_duplicates_sum(o):
    rng = np.random.default_rng(7)
    g = random_csr(rng, 30, 20, max_deg=8, weighted=False)
    B = rng.standard_normal((20, 6)).astype(np.float32)
    ones = np.ones(g.nnz, np.float32)
    for red in ("sum", "mean", "max"):
        C0, A0, _ = o.spmm(g.rowptr, g.col, None, B, red)
        C1, A1, _ = o.spmm(g.rowptr, g.col, ones, B, red)
        assert np.array_equal(C0, C1)
        if red == "max":
            assert np.array_equal(A0, A1)
    # a duplicated entry counts twice: same as a single entry with value 2
    g2 = gen.from_rows("d", 1, 3, [[1, 1, 2]], [[1.0, 1.0, 1.0]])
    g3 = gen.from_rows("d", 1, 3, [[1, 2]], [[2.0, 1.0]])
    B = np.array([[0.0], [1.5], [-4.0]], np.float32)
    assert np.array_equal(o.spmm(g2.rowptr, g2.col, g2.val, B, "sum")[0],
                          o.spmm(g3.rowptr, g3.col, g3.val, B, "sum")[0])
    # mean divides by the count of stored entries (3 here), not by distinct columns
    assert o.spmm(g2.rowptr, g2.col, g2.val, B, "mean")[0][0, 0] == np.float32(-1.0 / 3.0)


def pin_row_subset_matches_full(o):
    g = gen.erdos_renyi(200, 150, 5, seed=9)
    B = gen.features(150, 11, seed=9)
    rows = np.array([199, 0, 17, 17, 63])
    for red in ("sum", "mean", "max"):
        Cf, Af, Tf = o.spmm(g.rowptr, g.col, g.val, B, red)
        Cs, As, Ts = o.spmm(g.rowptr, g.col, g.val, B, red, rows=rows)
        assert np.array_equal(Cs, Cf[rows])
        if red == "max":
            assert np.array_equal(As, Af[rows])
        else:
            assert np.array_equal(Ts, Tf[rows])


def _relu(x):
    return np.where(x > 0, x, np.float32(0.0)).astype(np.float32)


def pin_epilogue_identity_graph(o):
    # identity: R = B exactly, so act(R + bias) is one fp64 addition rounded once
    M, N = 40, 9
    g = gen.from_rows("eye", M, M, [[i] for i in range(M)])
    B = gen.features(M, N, seed=5)
    bias = gen.features(1, N, seed=6)[0]
    want = (B.astype(np.float64) + bias.astype(np.float64)).astype(np.float32)
    for red in ("sum", "mean", "max"):
        C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, red, bias=bias)
        assert np.array_equal(C, want), red
        C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, red, bias=bias, act="relu")
        assert np.array_equal(C, _relu(want)), red
        if red == "max":
            assert np.array_equal(A, np.repeat(np.arange(M, dtype=np.int32)[:, None], N, 1))
        C, _, _ = o.spmm(g.rowptr, g.col, g.val, B, red, act="relu")
        assert np.array_equal(C, _relu(B)), red


def pin_epilogue_ring_graph_and_empty_rows(o):
    # ring: R = B[i-1] + B[i+1] (exact in fp64), mean R / 2 (exact); empty rows R = 0
    M, N = 31, 6
    rows = [[(i - 1) % M, (i + 1) % M] if i % 5 else [] for i in range(M)]
    g = gen.from_rows("ring_holes", M, M, rows)
    B = gen.features(M, N, seed=7)
    bias = gen.features(1, N, seed=8)[0].astype(np.float64)
    B64 = B.astype(np.float64)
    S = np.zeros((M, N))
    for i in range(M):
        if rows[i]:
            S[i] = B64[(i - 1) % M] + B64[(i + 1) % M]
    for red, R in (("sum", S), ("mean", S / 2)):
        want = _relu((R + bias).astype(np.float32))
        C, _, _ = o.spmm(g.rowptr, g.col, g.val, B, red, bias=bias.astype(np.float32), act="relu")
        assert np.array_equal(C, want), red
    C, A, _ = o.spmm(g.rowptr, g.col, g.val, B, "max", bias=bias.astype(np.float32), act="relu")
    empty = np.array([not r for r in rows])
    assert np.array_equal(C[empty], np.tile(_relu(bias.astype(np.float32)), (int(empty.sum()), 1)))
    assert np.all(A[empty] == -1)


def pin_descriptors_closed_forms(o):
    d = o.descriptors(np.arange(0, 41, 4, dtype=np.int32))      # 10 rows of degree 4
    assert d["M"] == 10 and d["nnz"] == 40 and d["dbar"] == 4.0 and d["cv"] == 0.0
    assert d["d_max"] == 4 and d["n_empty"] == 0
    rp = np.array([0, 0, 2, 2, 4, 4, 6, 6, 8], np.int32)               # degrees 0,2,0,2,...
    d = o.descriptors(rp)
    assert d["dbar"] == 1.0 and abs(d["cv"] - 1.0) < 1e-15 and d["n_empty"] == 4
    rp = np.array([0, 0, 0, 9], np.int32)                              # degrees 0,0,9
    d = o.descriptors(rp)
    assert d["dbar"] == 3.0 and abs(d["cv"] - np.sqrt(2.0)) < 1e-15 and d["d_max"] == 9
    d = o.descriptors(np.zeros(1, np.int32))
    assert d["M"] == 0 and d["nnz"] == 0
    with pytest.raises(ValueError):
        o.descriptors(np.array([0, 3, 2], np.int32))


def pin_descriptors_against_degree_statistics(o):
    g = gen.rmat(scale=11, edge_factor=8, seed=2)
    d = o.descriptors(g.rowptr)
    deg = g.degrees().astype(np.float64)
    assert d["nnz"] == g.nnz and d["d_max"] == deg.max()
    assert abs(d["dbar"] - deg.mean()) <= 1e-12 * deg.mean()
    assert abs(d["cv"] - deg.std() / deg.mean()) <= 1e-9


PINS = {name[4:]: fn for name, fn in sorted(globals().items()) if name.startswith("pin_")}


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(name):
    PINS[name](oracle._default())


# planted mistake -> a description; each must be rejected by at least one pin
PLANTS = {1: "drops the last term of each row", 2: "reads the wrong B row (col + 1)",
          3: "transposed B operand", 4: "max ties go to the larger column",
          5: "mean divides by d + 1", 6: "ReLU applied before the bias"}


@pytest.mark.parametrize("n", sorted(PLANTS))
def test_planted_mistake_is_caught(n, tmp_path):
    bad = oracle.planted(n, str(tmp_path))
    failed = []
    for name, fn in PINS.items():
        try:
            fn(bad)
        except AssertionError:
            failed.append(name)
    assert failed, f"no pin rejects planted mistake {n}: {PLANTS[n]}"
