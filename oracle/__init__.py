"""CPU oracle for CSR SpMM (sum, mean, max + argmax) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it; the two
share no code. The arithmetic lives in ``spmm_oracle.c`` (fp64 accumulation per
row in CSR order); this module compiles it with gcc on first use and wraps it
with ctypes.

Semantics (graph-spmm model card, "API" and "Correctness"; ParamSpMM
section 2, Algorithm 1):

* ``sum``  C[i,k] = sum over stored entries p of row i of a_p * B[col_p, k]
* ``mean`` the sum divided by the number of stored entries of row i; empty -> 0
* ``max``  max over the fp32-rounded products, ties to the smallest column;
           empty -> (0, -1)

``T`` (returned for sum/mean) is sum_p |a_p * B[col_p, k]|, the scale of the
tolerance |err| <= 1e-5 * T + 1e-6.

Backward (graph-spmm card, "Requirements and limits" and "API"): ``transpose``
builds A^T in CSR (stable by row; optionally each value divided by its row's
degree, for the mean), so that the sum / mean backward is a product with it;
``maxpool_backward`` routes dC[i, k] to the forward argmax column, through the
one stored entry (of a duplicated pair) whose product won.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmm_oracle.c")
_LIB = os.path.join(_HERE, "libspmm_oracle.so")
_lock = threading.Lock()
_lib = None

REDUCE = {"sum": 0, "mean": 1, "max": 2}
ACT = {"none": 0, "relu": 1}


class _Desc(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("nnz", ctypes.c_int64), ("d_max", ctypes.c_int64),
                ("n_empty", ctypes.c_int64), ("dbar", ctypes.c_double), ("cv", ctypes.c_double)]


def _compile(out: str, defines=()) -> None:
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]
    cmd += [f"-D{d}" for d in defines]
    subprocess.run(cmd + ["-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile the oracle library (plain C, OpenMP, no FP contraction)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
        if force or not fresh:
            _compile(_LIB)
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one build of spmm_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_spmm_rows.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int, p, i64, p, p, p]
        lib.oracle_spmm_rows.restype = ctypes.c_int
        lib.oracle_spmm_rows_ex.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int, p, ctypes.c_int,
                                            p, i64, p, p, p]
        lib.oracle_spmm_rows_ex.restype = ctypes.c_int
        lib.oracle_descriptors.argtypes = [i64, p, ctypes.POINTER(_Desc)]
        lib.oracle_descriptors.restype = ctypes.c_int
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_transpose.argtypes = [i64, i64, p, p, p, ctypes.c_int, p, p, p]
        lib.oracle_transpose.restype = ctypes.c_int
        lib.oracle_maxpool_backward.argtypes = [i64, i64, i64, p, p, p, p, p, p, p]
        lib.oracle_maxpool_backward.restype = ctypes.c_int
        self.lib = lib

    def threads(self) -> int:
        return int(self.lib.oracle_threads())

    def spmm(self, rowptr, col, val, B, reduce: str, rows=None, K=None, bias=None, act="none"):
        rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
        col = np.ascontiguousarray(col, dtype=np.int32)
        val = None if val is None else np.ascontiguousarray(val, dtype=np.float32)
        B = np.ascontiguousarray(B, dtype=np.float32)
        if B.ndim != 2:
            raise ValueError("B must be 2-D")
        M = len(rowptr) - 1
        K = B.shape[0] if K is None else K
        N = B.shape[1]
        if rows is None:
            R, rows_arr = M, None
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            R = len(rows_arr)
        red = REDUCE[reduce]
        C = np.empty((R, N), dtype=np.float32)
        A = np.empty((R, N), dtype=np.int32) if red == 2 else None
        T = np.empty((R, N), dtype=np.float32) if red != 2 else None
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.float32)
            if bias.shape != (N,):
                raise ValueError("bias must hold N values")
        rc = self.lib.oracle_spmm_rows_ex(M, K, N, _ptr(rowptr), _ptr(col), _ptr(val), _ptr(B), red,
                                          _ptr(bias), ACT[act], _ptr(rows_arr), R, _ptr(C),
                                          _ptr(A), _ptr(T))
        if rc != 0:
            raise ValueError("oracle_spmm_rows rejected its arguments")
        return C, A, T

    def descriptors(self, rowptr) -> dict:
        rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
        d = _Desc()
        if self.lib.oracle_descriptors(len(rowptr) - 1, _ptr(rowptr), ctypes.byref(d)) != 0:
            raise ValueError("invalid row pointers")
        return dict(M=d.M, nnz=d.nnz, d_max=d.d_max, n_empty=d.n_empty, dbar=d.dbar, cv=d.cv)


    def transpose(self, rowptr, col, val, K, scale_mean=False):
        """A^T in CSR: (rowptrT [K+1], colT [nnz], valT [nnz] or None)."""
        rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
        col = np.ascontiguousarray(col, dtype=np.int32)
        val = None if val is None else np.ascontiguousarray(val, dtype=np.float32)
        M = len(rowptr) - 1
        nnz = int(rowptr[-1])
        rT = np.empty(K + 1, np.int32)
        cT = np.empty(nnz, np.int32)
        vT = np.empty(nnz, np.float32) if (val is not None or scale_mean) else None
        if self.lib.oracle_transpose(M, K, _ptr(rowptr), _ptr(col), _ptr(val), int(scale_mean),
                                     _ptr(rT), _ptr(cT), _ptr(vT)) != 0:
            raise ValueError("oracle_transpose rejected its arguments")
        return rT, cT, vT

    def maxpool_backward(self, rowptr, col, val, argmax, dC, K, B=None):
        """dB [K, N] of the max reduction, given the forward argmax, dC [M, N]
        and, for a weighted A, the forward's B [K, N] (it decides which stored
        copy of a duplicated pair won)."""
        rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
        col = np.ascontiguousarray(col, dtype=np.int32)
        val = None if val is None else np.ascontiguousarray(val, dtype=np.float32)
        argmax = np.ascontiguousarray(argmax, dtype=np.int32)
        dC = np.ascontiguousarray(dC, dtype=np.float32)
        B = None if B is None else np.ascontiguousarray(B, dtype=np.float32)
        M, N = dC.shape
        if B is not None and B.shape != (K, N):
            raise ValueError("B must be [K, N]")
        dB = np.empty((K, N), np.float32)
        if self.lib.oracle_maxpool_backward(M, K, N, _ptr(rowptr), _ptr(col), _ptr(val), _ptr(B),
                                            _ptr(argmax), _ptr(dC), _ptr(dB)) != 0:
            raise ValueError("oracle_maxpool_backward rejected its arguments")
        return dB


def planted(n: int, out_dir: str) -> Oracle:
    """A build with planted mistake n (1..5), for the tests that check the pins."""
    out = os.path.join(out_dir, f"libspmm_oracle_plant{n}.so")
    _compile(out, [f"ORACLE_PLANT={n}"])
    return Oracle(out)


def _default() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def threads() -> int:
    return _default().threads()


def spmm(rowptr, col, val, B, reduce: str, rows=None, K=None, bias=None, act="none"):
    """Oracle SpMM. Returns (C float32 [R,N], argmax int32 [R,N] or None, T float32 [R,N] or None).

    ``rows`` selects output rows (int64 array); None means all M rows. ``bias``
    (float32 [N]) and ``act`` ("none" or "relu") give the fused epilogue
    act(R + bias); T is the tolerance scale of the reduction alone.
    """
    return _default().spmm(rowptr, col, val, B, reduce, rows, K, bias, act)


def descriptors(rowptr) -> dict:
    """M, nnz, d_max, n_empty, dbar = nnz/M, cv = std(d)/mean(d) over all rows."""
    return _default().descriptors(rowptr)


def transpose(rowptr, col, val, K, scale_mean=False):
    """A^T in CSR (stable by row); scale_mean divides each value by its row's degree."""
    return _default().transpose(rowptr, col, val, K, scale_mean)


def maxpool_backward(rowptr, col, val, argmax, dC, K, B=None):
    """Gradient of the max reduction with respect to B: dC[i, k] times the
    weight of the stored entry that won the forward maximum (B is needed when
    A is weighted)."""
    return _default().maxpool_backward(rowptr, col, val, argmax, dC, K, B)
