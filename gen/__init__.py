"""Seeded synthetic inputs for CSR SpMM: graph adjacencies in CSR and dense features.

This module builds inputs only. It holds none of the product's arithmetic
(no sum, mean or max over neighbours), so both the CPU oracle and the CUDA
path take their inputs from here and share nothing else.

Every array comes from its own numpy PCG64 stream, keyed by
(seed, graph family, array name, sizes), so a graph and its features are
reproducible and independent of the order in which they are made.

Graph families (the five workload shapes the engine is measured on, plus
scaled-down versions of each for parity tests):

* ``erdos_renyi``   -- every row draws ``deg`` distinct uniform columns, val U(0,1).
* ``knn_local``     -- every row draws ``deg`` distinct columns uniformly within
                       +-``window`` of its own id (self excluded), val absent.
* ``rmat``          -- R-MAT edge recursion (a, b, c, d), duplicates removed,
                       ids permuted, val = 1/deg(row).
* ``community``     -- blocks of consecutive ids; intra-block Bernoulli(p) edges
                       (self excluded) plus ``n_inter`` distinct uniform columns
                       outside the block, val U(0,1).
* ``chung_lu``      -- expected degrees w_i = c (i+1)^(-1/(gamma-1)) capped at
                       ``cap``, c chosen so mean(w) = ``mean``; row i draws
                       Poisson(w_i) distinct columns with probability
                       proportional to w_j; ids permuted; val U(0,1).

CSR conventions: ``rowptr`` int32 [M+1], ``col`` int32 [nnz] ascending within a
row, ``val`` float32 [nnz] or None (unweighted).
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

__all__ = [
    "Graph", "rng_for", "features", "uniform01", "csr_from_keys",
    "erdos_renyi", "knn_local", "rmat", "community", "chung_lu",
    "from_rows", "config", "CONFIGS",
]


@dataclasses.dataclass
class Graph:
    name: str
    M: int
    K: int
    rowptr: np.ndarray          # int32 [M+1]
    col: np.ndarray             # int32 [nnz]
    val: np.ndarray | None      # float32 [nnz] or None

    @property
    def nnz(self) -> int:
        return int(self.rowptr[-1])

    def degrees(self) -> np.ndarray:
        return np.diff(self.rowptr.astype(np.int64))


def rng_for(seed: int, *tags) -> np.random.Generator:
    """Independent PCG64 stream for (seed, tags...); string tags are hashed with CRC32."""
    words = [int(seed) & 0xFFFFFFFF]
    for t in tags:
        if isinstance(t, str):
            words.append(zlib.crc32(t.encode()) & 0xFFFFFFFF)
        else:
            v = int(t)
            words.append(v & 0xFFFFFFFF)
            words.append((v >> 32) & 0xFFFFFFFF)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def uniform01(rng: np.random.Generator, n: int) -> np.ndarray:
    """U[0,1) in float32 from a 24-bit integer draw (every value exactly representable)."""
    return (rng.integers(0, 1 << 24, size=n, dtype=np.int64).astype(np.float32)
            * np.float32(1.0 / (1 << 24)))


def features(K: int, N: int, seed: int = 0, tag: str = "B") -> np.ndarray:
    """Dense K x N float32 feature matrix, N(0,1), row-major."""
    rng = rng_for(seed, "features", tag, K, N)
    return rng.standard_normal(size=(K, N), dtype=np.float32)


def csr_from_keys(keys: np.ndarray, M: int, K: int):
    """Sorted (row*K + col) int64 keys -> (rowptr int32 [M+1], col int32 [nnz])."""
    rows = keys // K
    col = (keys - rows * K).astype(np.int32)
    counts = np.bincount(rows, minlength=M)
    rowptr = np.zeros(M + 1, dtype=np.int64)
    np.cumsum(counts, out=rowptr[1:])
    if rowptr[-1] >= 2**31:
        raise ValueError("nnz does not fit int32 row pointers")
    return rowptr.astype(np.int32), col


def from_rows(name: str, M: int, K: int, rows, val_rows=None) -> Graph:
    """CSR from explicit per-row column lists (kept in the given order, duplicates kept)."""
    rowptr = np.zeros(M + 1, dtype=np.int64)
    for i, r in enumerate(rows):
        rowptr[i + 1] = rowptr[i] + len(r)
    col = np.array([c for r in rows for c in r], dtype=np.int32)
    val = None
    if val_rows is not None:
        val = np.array([v for r in val_rows for v in r], dtype=np.float32)
    return Graph(name, M, K, rowptr.astype(np.int32), col, val)


def _sorted_unique(x):
    """np.unique for int64 keys via one sort (np.unique is far slower on large arrays)."""
    x = np.sort(x)
    if len(x) < 2:
        return x
    keep = np.empty(len(x), dtype=bool)
    keep[0] = True
    np.not_equal(x[1:], x[:-1], out=keep[1:])
    return x[keep]


def _fill_distinct(counts, draw, K, exclude=None):
    """Per row r, counts[r] distinct columns: draw(rows) gives candidate columns for
    the given row ids; exclude(rows, cols) marks forbidden pairs.

    Every slot is drawn once; the slots lost to repeats or exclusions are drawn
    again (only those) until each row holds counts[r] distinct columns.
    Returns sorted int64 keys row*K + col.
    """
    M = len(counts)
    counts = counts.astype(np.int64)
    rows = np.repeat(np.arange(M, dtype=np.int64), counts)
    cols = draw(rows)
    if exclude is not None:
        keep = ~exclude(rows, cols)
        rows, cols = rows[keep], cols[keep]
    S = _sorted_unique(rows * K + cols)
    del rows, cols
    have = np.bincount(S // K, minlength=M)
    A = np.empty(0, dtype=np.int64)
    missing = counts - have
    while missing.sum() > 0:
        r = np.repeat(np.arange(M, dtype=np.int64), missing)
        c = draw(r)
        if exclude is not None:
            keep = ~exclude(r, c)
            r, c = r[keep], c[keep]
        k = r * K + c
        for ref in (S, A):
            if len(ref) and len(k):
                pos = np.minimum(np.searchsorted(ref, k), len(ref) - 1)
                k = k[ref[pos] != k]
        k = _sorted_unique(k)
        A = np.sort(np.concatenate([A, k]))
        missing = counts - have - np.bincount(A // K, minlength=M)
    if len(A):
        S = np.insert(S, np.searchsorted(S, A), A)
    return S


def _distinct_in_window(rng, lo, hi, deg, exclude_col):
    """Row r: deg[r] distinct ints uniform in [lo[r], hi[r]], never exclude_col[r]."""
    span = (hi - lo + 1).astype(np.int64)
    inside = ((exclude_col >= lo) & (exclude_col <= hi)).astype(np.int64)
    if np.any(span - inside < deg):
        raise ValueError("window too small for the requested degree")
    K = int(hi.max()) + 1

    def draw(rows):
        return lo[rows] + (rng.random(len(rows)) * span[rows]).astype(np.int64)

    def excl(rows, cols):
        return cols == exclude_col[rows]

    return _fill_distinct(deg, draw, K, excl), K


def erdos_renyi(M: int = 2048, K: int = 2048, deg: int = 8, seed: int = 0,
                weighted: bool = True) -> Graph:
    rng = rng_for(seed, "erdos_renyi", M, K, deg)
    lo = np.zeros(M, dtype=np.int64)
    hi = np.full(M, K - 1, dtype=np.int64)
    keys, Kw = _distinct_in_window(rng, lo, hi, np.full(M, deg), np.full(M, -1, dtype=np.int64))
    rowptr, col = csr_from_keys(keys, M, Kw)
    val = uniform01(rng_for(seed, "erdos_renyi/val", M, K, deg), len(col)) if weighted else None
    return Graph(f"er_M{M}_d{deg}", M, K, rowptr, col, val)


def knn_local(M: int = 1 << 20, deg: int = 10, window: int = 512, seed: int = 0,
              weighted: bool = False) -> Graph:
    rng = rng_for(seed, "knn_local", M, deg, window)
    i = np.arange(M, dtype=np.int64)
    lo = np.maximum(0, i - window)
    hi = np.minimum(M - 1, i + window)
    keys, Kw = _distinct_in_window(rng, lo, hi, np.full(M, deg), i)
    rowptr, col = csr_from_keys(keys, M, Kw)
    val = uniform01(rng_for(seed, "knn_local/val", M, deg, window), len(col)) if weighted else None
    return Graph(f"knn_M{M}_d{deg}_w{window}", M, M, rowptr, col, val)


def _permutation(seed, tag, n):
    return rng_for(seed, tag, n).permutation(n).astype(np.int64)


def rmat(scale: int = 20, edge_factor: int = 16, a: float = 0.57, b: float = 0.19,
         c: float = 0.19, seed: int = 0, permute: bool = True) -> Graph:
    """R-MAT: each of edge_factor * 2^scale edges descends `scale` quadrant levels."""
    n = 1 << scale
    E = edge_factor * n
    rng = rng_for(seed, "rmat", scale, edge_factor)
    src = np.zeros(E, dtype=np.int64)
    dst = np.zeros(E, dtype=np.int64)
    ab, abc = a + b, a + b + c
    for _ in range(scale):
        u = rng.random(E)
        sbit = u >= ab                               # quadrants c, d: lower half
        dbit = ((u >= a) & (u < ab)) | (u >= abc)    # quadrants b, d: right half
        src = (src << 1) | sbit
        dst = (dst << 1) | dbit
    if permute:
        perm = _permutation(seed, "rmat/perm", n)
        src = perm[src]
        dst = perm[dst]
    keys = _sorted_unique(src * n + dst)
    del src, dst
    rowptr, col = csr_from_keys(keys, n, n)
    deg = np.diff(rowptr.astype(np.int64))
    inv = np.zeros(n, dtype=np.float32)
    nz = deg > 0
    inv[nz] = (1.0 / deg[nz]).astype(np.float32)
    val = np.repeat(inv, deg)
    return Graph(f"rmat_s{scale}_ef{edge_factor}", n, n, rowptr, col, val)


def community(n_comm: int = 256, comm_size: int = 256, p: float = 0.2, n_inter: int = 5,
              seed: int = 0) -> Graph:
    M = n_comm * comm_size
    rng = rng_for(seed, "community", n_comm, comm_size)
    # intra-block Bernoulli(p) over the other members of the row's block
    hit = rng.random((M, comm_size)) < p
    hit[np.arange(M), np.arange(M) % comm_size] = False
    r_in, c_in = np.nonzero(hit)
    del hit
    keys_in = r_in.astype(np.int64) * M + (r_in // comm_size) * comm_size + c_in
    # n_inter distinct uniform columns outside the block: draw in [0, M - comm_size)
    # and shift the draws at or past the block start over the block
    rng2 = rng_for(seed, "community/inter", n_comm, comm_size)
    lo = np.zeros(M, dtype=np.int64)
    hi = np.full(M, M - comm_size - 1, dtype=np.int64)
    kb, Kw = _distinct_in_window(rng2, lo, hi, np.full(M, n_inter), np.full(M, -1, dtype=np.int64))
    r_out = kb // Kw
    c_out = kb - r_out * Kw
    blk0 = (r_out // comm_size) * comm_size
    c_out = np.where(c_out >= blk0, c_out + comm_size, c_out)
    keys = np.sort(np.concatenate([keys_in, r_out * M + c_out]))
    rowptr, col = csr_from_keys(keys, M, M)
    val = uniform01(rng_for(seed, "community/val", n_comm, comm_size), len(col))
    return Graph(f"community_{n_comm}x{comm_size}", M, M, rowptr, col, val)


def chung_lu_weights(M: int, gamma: float = 2.1, mean: float = 25.0, cap: float = 1e5):
    """w_i = min(c (i+1)^(-1/(gamma-1)), cap), c found by bisection so that mean(w) = mean."""
    x = np.arange(1, M + 1, dtype=np.float64) ** (-1.0 / (gamma - 1.0))
    lo, hi = 0.0, cap * 2.0 + mean * M
    for _ in range(64):
        mid = 0.5 * (lo + hi)
        if np.minimum(mid * x, cap).mean() < mean:
            lo = mid
        else:
            hi = mid
    return np.minimum(hi * x, cap)


def chung_lu(M: int = 1 << 22, gamma: float = 2.1, mean: float = 25.0, cap: float = 1e5,
             seed: int = 0, permute: bool = True) -> Graph:
    """Rows and columns are drawn in the weight order, then relabelled by one permutation."""
    w = chung_lu_weights(M, gamma, mean, cap)
    rng = rng_for(seed, "chung_lu", M, int(mean * 1000), int(cap))
    deg = np.minimum(rng.poisson(w).astype(np.int64), M)
    cdf = np.cumsum(w)
    total = cdf[-1]
    perm = _permutation(seed, "chung_lu/perm", M) if permute else np.arange(M, dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(M, dtype=np.int64)

    def draw(rows):
        # inverse-CDF draws; the queries are sorted first (a sorted searchsorted is
        # cache friendly) and handed to the slots in a random order afterwards
        n = len(rows)
        q = np.sort(rng.random(n) * total)
        j = np.minimum(np.searchsorted(cdf, q, side="right"), M - 1)
        out = np.empty(n, dtype=np.int64)
        out[rng.permutation(n)] = perm[j]
        return out

    deg_new = np.empty_like(deg)
    deg_new[perm] = deg                      # new row perm[i] carries old row i's degree
    keys = _fill_distinct(deg_new, draw, M)
    rowptr, col = csr_from_keys(keys, M, M)
    del keys
    val = uniform01(rng_for(seed, "chung_lu/val", M), len(col))
    return Graph(f"chung_lu_M{M}", M, M, rowptr, col, val)


# The five measured workloads: (graph builder, feature widths, reductions).
CONFIGS = {
    1: dict(name="erdos_renyi_2k", build=lambda s=0: erdos_renyi(2048, 2048, 8, s),
            N=(32,), reduce=("sum", "mean", "max")),
    2: dict(name="knn_1M", build=lambda s=0: knn_local(1 << 20, 10, 512, s),
            N=(16, 64), reduce=("sum", "mean")),
    3: dict(name="rmat_s20", build=lambda s=0: rmat(20, 16, 0.57, 0.19, 0.19, s),
            N=(64, 128, 256), reduce=("sum", "max")),
    4: dict(name="community_64k", build=lambda s=0: community(256, 256, 0.2, 5, s),
            N=(128, 512), reduce=("sum",)),
    5: dict(name="chung_lu_4M", build=lambda s=0: chung_lu(1 << 22, 2.1, 25.0, 1e5, s),
            N=(16, 32, 64, 128, 256), reduce=("sum", "mean", "max")),
}


def config(cid: int, seed: int = 0) -> Graph:
    return CONFIGS[cid]["build"](seed)
