"""GB300 CSR SpMM engine: Python binding of libspmm.so (include/spmm.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory and the current stream. If the
library has not been built the import fails loudly; there is no CPU fallback.

The API mirrors the graph-spmm model card ("API"):

* ``spmm_sum / spmm_mean / spmm_max / spmm(rowptr, col, val, mat, reduce)``
* ``SparseAdj(rowptr, col, val)`` -- a CSR adjacency held once (one plan) and
  applied many times: ``adj @ x``, ``adj.reduce(x, "mean")``,
  ``values, argmax = adj.reduce(x, "max")``.

The C-ABI calls are exposed under their own names as well
(``spmm_plan_create``, ``spmm_run``, ...), taking raw device pointers.

Tensors: ``rowptr`` int32 [M+1], ``col`` int32 [nnz], ``val`` float32 [nnz] or
None (unweighted), ``mat`` float32 [K, N] row-major; all on the same CUDA device.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH
from ._build import build as build_library

__all__ = [
    "SparseAdj", "SpmmError", "spmm", "spmm_sum", "spmm_mean", "spmm_max",
    "spmm_plan_create", "spmm_run", "spmm_plan_describe", "spmm_plan_destroy",
    "spmm_plan_reserve", "spmm_plan_validate_cols", "spmm_plan_sync", "spmm_plan_set_family",
    "spmm_route", "spmm_default_t_split", "spmm_status_string", "spmm_launch_count",
    "spmm_run_noalloc", "spmm_transpose", "spmm_maxpool_backward", "spmm_run_ex", "ACT",
    "spmm_check_wait_timeout", "spmm_plan_create_range", "spmm_partition_rows",
    "spmm_plan_prepare_blocks",
    "PlanInfo", "REDUCE", "FAMILY", "lib", "build_library",
]

REDUCE = {"sum": 0, "mean": 1, "max": 2}
ACT = {None: 0, "none": 0, "relu": 1}
FAMILY = {"auto": -1, "rowgroup": 0, "warprow": 1, "coltile": 2, "window": 3, "block": 4,
          "segment": 5, "gather": 6, "stream": 7}
STATUS = {0: "SPMM_OK", 1: "SPMM_ERR_INVALID_ARG", 2: "SPMM_ERR_INVALID_INPUT", 3: "SPMM_ERR_OOM",
          4: "SPMM_ERR_CUDA", 5: "SPMM_ERR_UNSUPPORTED", 6: "SPMM_ERR_TIMEOUT"}


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("nnz", ctypes.c_int64),
        ("d_max", ctypes.c_int64), ("n_empty", ctypes.c_int64),
        ("dbar", ctypes.c_double), ("cv", ctypes.c_double),
        ("t_split", ctypes.c_int64), ("chunk", ctypes.c_int64),
        ("n_heavy", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
        ("N", ctypes.c_int64), ("reduce", ctypes.c_int32), ("family", ctypes.c_int32),
        ("vec", ctypes.c_int32), ("lanes", ctypes.c_int32), ("rows_per_warp", ctypes.c_int32),
        ("col_tiles", ctypes.c_int32), ("launches", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("band_w", ctypes.c_int64), ("band_cover", ctypes.c_double),
        ("window_rows", ctypes.c_int32), ("window_ctas", ctypes.c_int32),
        ("window_smem", ctypes.c_int64), ("window_chunks", ctypes.c_int32),
        ("rows_sorted", ctypes.c_int32), ("blk_intra", ctypes.c_int64),
        ("row0", ctypes.c_int64),
        ("seg_tiles", ctypes.c_int64), ("seg_warps", ctypes.c_int32),
        ("seg_chunks", ctypes.c_int32), ("block_bytes", ctypes.c_int64),
        ("gather_bytes", ctypes.c_int64), ("gather_ctas", ctypes.c_int32),
        ("stream_ranges", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["family_name"] = {v: k for k, v in FAMILY.items()}.get(d["family"], "?")
        return d


class SpmmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({spmm_status_string(status)})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()'); there is no CPU fallback")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER
    sigs = {
        "spmm_plan_create": ([vp, i64, i64, vp, P(vp)], i32),
        "spmm_plan_create_range": ([vp, i64, i64, i64, vp, P(vp)], i32),
        "spmm_partition_rows": ([vp, i64, i32, i64, P(ctypes.c_int64)], i32),
        "spmm_run": ([vp, vp, vp, vp, i64, i32, vp, vp, vp], i32),
        "spmm_run_ex": ([vp, vp, vp, vp, i64, i32, vp, i32, vp, vp, vp], i32),
        "spmm_plan_reserve": ([vp, i64, i32], i32),
        "spmm_plan_validate_cols": ([vp, vp, vp], i32),
        "spmm_plan_sync": ([vp, vp], i32),
        "spmm_plan_prepare_blocks": ([vp, vp, vp, vp], i32),
        "spmm_plan_describe": ([vp, i64, i32, P(PlanInfo)], i32),
        "spmm_plan_set_family": ([vp, i32, i64], i32),
        "spmm_route": ([P(PlanInfo), i64, i32, i32, i32, i32, P(PlanInfo)], i32),
        "spmm_default_t_split": ([i64, i64, i32], i64),
        "spmm_plan_destroy": ([vp], i32),
        "spmm_status_string": ([i32], ctypes.c_char_p),
        "spmm_launch_count": ([], ctypes.c_uint64),
        "spmm_run_noalloc": ([vp, vp, vp, vp, i64, i64, i64, i32, vp, vp, vp], i32),
        "spmm_transpose": ([vp, vp, vp, i32, vp, vp, vp, vp], i32),
        "spmm_check_wait_timeout": ([vp, i64, vp], i32),
        "spmm_maxpool_backward": ([vp, vp, vp, vp, vp, vp, i64, vp, vp], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


lib = _load()


def _check(status: int, what: str):
    if status != 0:
        raise SpmmError(status, what)


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) or None


# ---------------------------------------------------------------- raw C ABI
def spmm_status_string(status: int) -> str:
    return lib.spmm_status_string(int(status)).decode()


def spmm_launch_count() -> int:
    return int(lib.spmm_launch_count())


def spmm_default_t_split(M: int, nnz: int, num_sms: int) -> int:
    return int(lib.spmm_default_t_split(M, nnz, num_sms))


def spmm_plan_create_range(rowptr_ptr: int, row_begin: int, row_end: int, K: int,
                           stream=None) -> int:
    """Plan for rows [row_begin, row_end) of the matrix whose whole rowptr is given."""
    out = ctypes.c_void_p()
    _check(lib.spmm_plan_create_range(rowptr_ptr, row_begin, row_end, K, _stream_handle(stream),
                                      ctypes.byref(out)), "spmm_plan_create_range")
    return out.value


def spmm_partition_rows(rowptr, parts: int, align_rows: int = 1) -> list:
    """Row bounds [b_0 = 0, ..., b_parts = M] of `parts` contiguous ranges balanced
    by entries + rows. ``rowptr``: a host array (numpy or CPU tensor; a CUDA
    tensor is copied to the host first)."""
    import numpy as np
    if hasattr(rowptr, "detach"):
        rowptr = rowptr.detach().cpu().numpy()
    rp = np.ascontiguousarray(rowptr, dtype=np.int32)
    if rp.ndim != 1 or rp.size < 1:
        raise ValueError("rowptr must be a 1-D array of M+1 entries")
    if parts < 1:
        raise ValueError("parts must be >= 1")
    bounds = (ctypes.c_int64 * (parts + 1))()
    _check(lib.spmm_partition_rows(rp.ctypes.data, rp.size - 1, parts, align_rows, bounds),
           "spmm_partition_rows")
    return [int(b) for b in bounds]


def spmm_plan_create(rowptr_ptr: int, M: int, K: int, stream=None) -> int:
    out = ctypes.c_void_p()
    _check(lib.spmm_plan_create(rowptr_ptr, M, K, _stream_handle(stream), ctypes.byref(out)),
           "spmm_plan_create")
    return out.value


def spmm_run(plan: int, col_ptr: int, val_ptr, B_ptr: int, N: int, reduce: int, C_ptr: int,
             argmax_ptr=None, stream=None) -> None:
    _check(lib.spmm_run(plan, col_ptr, val_ptr, B_ptr, N, reduce, C_ptr, argmax_ptr,
                        _stream_handle(stream)), "spmm_run")


def spmm_run_ex(plan: int, col_ptr: int, val_ptr, B_ptr: int, N: int, reduce: int, bias_ptr,
                act: int, C_ptr: int, argmax_ptr=None, stream=None) -> None:
    """spmm_run with the fused epilogue C = act(R + bias)."""
    _check(lib.spmm_run_ex(plan, col_ptr, val_ptr, B_ptr, N, reduce, bias_ptr, act, C_ptr,
                           argmax_ptr, _stream_handle(stream)), "spmm_run_ex")


def spmm_plan_reserve(plan: int, N: int, reduce: int) -> None:
    _check(lib.spmm_plan_reserve(plan, N, reduce), "spmm_plan_reserve")


def spmm_plan_validate_cols(plan: int, col_ptr: int, stream=None) -> None:
    _check(lib.spmm_plan_validate_cols(plan, col_ptr, _stream_handle(stream)),
           "spmm_plan_validate_cols")


def spmm_plan_prepare_blocks(plan: int, col_ptr: int, val_ptr, stream=None) -> None:
    """The BLOCK family's per-plan preparation (dense diagonal blocks split
    into TF32 hi/lo, and the entries outside them); synchronous."""
    _check(lib.spmm_plan_prepare_blocks(plan, col_ptr, val_ptr, _stream_handle(stream)),
           "spmm_plan_prepare_blocks")


def spmm_plan_sync(plan: int, stream=None) -> None:
    _check(lib.spmm_plan_sync(plan, _stream_handle(stream)), "spmm_plan_sync")


def spmm_plan_describe(plan: int, N: int, reduce: int) -> dict:
    info = PlanInfo()
    _check(lib.spmm_plan_describe(plan, N, reduce, ctypes.byref(info)), "spmm_plan_describe")
    return info.as_dict()


def spmm_plan_set_family(plan: int, family: int, t_split: int = 0) -> None:
    _check(lib.spmm_plan_set_family(plan, family, t_split), "spmm_plan_set_family")


def spmm_plan_destroy(plan: int) -> None:
    _check(lib.spmm_plan_destroy(plan), "spmm_plan_destroy")


def spmm_route(desc: dict, N: int, reduce: int, aligned: int = 3, num_sms: int = 152,
               family: int = -1) -> dict:
    """The router as a pure host function (no GPU needed).

    ``aligned``: bit 0 = B/C/argmax 16-byte aligned, bit 1 = col/val 16-byte aligned,
    bit 2 = no val array.
    """
    d = PlanInfo()
    for k in ("M", "K", "nnz", "d_max", "n_empty", "dbar", "cv", "t_split", "chunk",
              "n_heavy", "n_chunks", "band_w", "band_cover", "rows_sorted", "blk_intra",
              "row0", "seg_tiles"):
        if k in desc:
            setattr(d, k, desc[k])
    out = PlanInfo()
    _check(lib.spmm_route(ctypes.byref(d), N, reduce, int(aligned), num_sms, family,
                          ctypes.byref(out)), "spmm_route")
    return out.as_dict()


def spmm_run_noalloc(rowptr_ptr: int, col_ptr: int, val_ptr, B_ptr: int, M: int, K: int, N: int,
                     reduce: int, C_ptr: int, argmax_ptr=None, stream=None) -> None:
    """spmm_run without a plan and without device allocation (see include/spmm.h)."""
    _check(lib.spmm_run_noalloc(rowptr_ptr, col_ptr, val_ptr, B_ptr, M, K, N, reduce, C_ptr,
                                argmax_ptr, _stream_handle(stream)), "spmm_run_noalloc")


def spmm_transpose(plan: int, col_ptr, val_ptr, scale_mean: bool, rowptrT_ptr: int, colT_ptr,
                   valT_ptr, stream=None) -> None:
    """A^T in CSR (synchronous; see include/spmm.h)."""
    _check(lib.spmm_transpose(plan, col_ptr, val_ptr, 1 if scale_mean else 0, rowptrT_ptr,
                              colT_ptr, valT_ptr, _stream_handle(stream)), "spmm_transpose")


def spmm_check_wait_timeout(plan: int, limit_us: int, stream=None) -> int:
    """Run one bounded wait that nothing completes; returns the status (6 = timeout)."""
    return int(lib.spmm_check_wait_timeout(plan, limit_us, _stream_handle(stream)))


def spmm_maxpool_backward(planT: int, colT_ptr, valT_ptr, B_ptr, argmax_ptr, dC_ptr, N: int,
                          dB_ptr: int, stream=None) -> None:
    """Gradient of spmm_max with respect to B, through the plan of A^T (B_ptr:
    the forward's B, required for a weighted A)."""
    _check(lib.spmm_maxpool_backward(planT, colT_ptr, valT_ptr, B_ptr, argmax_ptr, dC_ptr, N,
                                     dB_ptr, _stream_handle(stream)), "spmm_maxpool_backward")


# ------------------------------------------------------------ tensor API
def _req(t, dtype, name, dev=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    return t


class SparseAdj:
    """A CSR adjacency held once (one plan) and applied many times."""

    def __init__(self, rowptr, col, val=None, num_cols: int | None = None,
                 validate: bool = True, rows: tuple | None = None):
        """``rows=(b, e)`` builds the product for rows [b, e) only: rowptr, col
        and val are the whole matrix's, and outputs have e - b rows."""
        import torch
        _req(rowptr, torch.int32, "rowptr")
        dev = rowptr.device
        _req(col, torch.int32, "col", dev)
        if val is not None:
            _req(val, torch.float32, "val", dev)
            if val.numel() != col.numel():
                raise ValueError("val and col differ in length")
        self.device = dev
        M_all = rowptr.numel() - 1
        if M_all < 0:
            raise ValueError("rowptr must hold M+1 entries")
        self.rows = (0, M_all) if rows is None else (int(rows[0]), int(rows[1]))
        if not 0 <= self.rows[0] <= self.rows[1] <= M_all:
            raise ValueError(f"rows {rows} outside [0, {M_all}]")
        self.M = self.rows[1] - self.rows[0]
        self.K = int(num_cols) if num_cols is not None else M_all
        self.rowptr, self.col, self.val = rowptr, col, val
        self._plan = None
        self._t = self._tmean = None
        with torch.cuda.device(dev):
            if rows is None:
                self._plan = spmm_plan_create(rowptr.data_ptr(), self.M, self.K)
            else:
                self._plan = spmm_plan_create_range(rowptr.data_ptr(), self.rows[0], self.rows[1],
                                                    self.K)
            info = spmm_plan_describe(self._plan, 0, 0)
            self.nnz = info["nnz"]
            if (rows is None and self.nnz != col.numel()) or \
                    (rows is not None and int(rowptr[self.rows[1]]) > col.numel()):
                self.close()
                raise ValueError(f"rowptr holds {self.nnz} entries for these rows but col "
                                 f"holds {col.numel()}")
            if validate:
                try:
                    spmm_plan_validate_cols(self._plan, col.data_ptr())
                except SpmmError:
                    self.close()
                    raise

    @property
    def plan(self) -> int:
        if self._plan is None:
            raise RuntimeError("SparseAdj is closed")
        return self._plan

    def describe(self, N: int, reduce: str = "sum") -> dict:
        return spmm_plan_describe(self.plan, N, REDUCE[reduce])

    def set_family(self, family: str = "auto", t_split: int = 0) -> None:
        import torch
        with torch.cuda.device(self.device):
            spmm_plan_set_family(self.plan, FAMILY[family], t_split)

    def reserve(self, N: int, reduce: str = "sum") -> None:
        import torch
        with torch.cuda.device(self.device):
            spmm_plan_reserve(self.plan, N, REDUCE[reduce])

    def reduce(self, mat, reduce: str = "sum", out=None, argmax=None, stream=None, bias=None,
               activation=None):
        """sum / mean -> C [M, N]; max -> (C, argmax int32 [M, N]).

        ``bias`` (float32 [N]) and ``activation`` (None or "relu") fuse the
        epilogue C = act(R + bias) into the same launch."""
        import torch
        if reduce not in REDUCE:
            raise ValueError(f"unknown reduce {reduce!r}")
        if activation not in ACT:
            raise ValueError(f"unknown activation {activation!r}")
        _req(mat, torch.float32, "mat", self.device)
        if mat.dim() != 2 or mat.shape[0] != self.K:
            raise ValueError(f"mat must be [{self.K}, N], got {tuple(mat.shape)}")
        N = mat.shape[1]
        if out is None:
            out = torch.empty((self.M, N), dtype=torch.float32, device=self.device)
        else:
            _req(out, torch.float32, "out", self.device)
            if tuple(out.shape) != (self.M, N):
                raise ValueError("out has the wrong shape")
        red = REDUCE[reduce]
        if red == 2:
            if argmax is None:
                argmax = torch.empty((self.M, N), dtype=torch.int32, device=self.device)
            else:
                _req(argmax, torch.int32, "argmax", self.device)
                if tuple(argmax.shape) != (self.M, N):
                    raise ValueError("argmax has the wrong shape")
        if bias is not None:
            _req(bias, torch.float32, "bias", self.device)
            if tuple(bias.shape) != (N,):
                raise ValueError(f"bias must be [{N}]")
        with torch.cuda.device(self.device):
            spmm_run_ex(self.plan, self.col.data_ptr(),
                        None if self.val is None else self.val.data_ptr(),
                        mat.data_ptr(), N, red, None if bias is None else bias.data_ptr(),
                        ACT[activation], out.data_ptr(), argmax.data_ptr() if red == 2 else None,
                        stream)
        return (out, argmax) if red == 2 else out

    def __matmul__(self, mat):
        return self.reduce(mat, "sum")

    def transpose(self, scale_mean: bool = False) -> "SparseAdj":
        """A^T as a new SparseAdj (K x M). With ``scale_mean`` the value of entry
        (i, j) is a_ij / d_i, so that ``adj.transpose(True) @ dC`` is the
        gradient of ``adj.reduce(B, "mean")`` with respect to B. For a row range
        (``rows=(b, e)``) the result is K x (e - b), its columns the range's
        local row numbers."""
        import torch
        nnz = self.nnz
        rowptrT = torch.empty(self.K + 1, dtype=torch.int32, device=self.device)
        colT = torch.empty(nnz, dtype=torch.int32, device=self.device)
        valT = (torch.empty(nnz, dtype=torch.float32, device=self.device)
                if (self.val is not None or scale_mean) else None)
        with torch.cuda.device(self.device):
            spmm_transpose(self.plan, self.col.data_ptr(),
                           None if self.val is None else self.val.data_ptr(), scale_mean,
                           rowptrT.data_ptr(), colT.data_ptr(),
                           None if valT is None else valT.data_ptr())
        return SparseAdj(rowptrT, colT, valT, num_cols=self.M)

    def maxpool_backward(self, argmax, grad, B=None, out=None, stream=None):
        """Called on A^T (from ``transpose()``): the gradient of the max
        reduction with respect to B, given its argmax [M, N], dC [M, N] and,
        for a weighted A, the forward's B [K, N] (which copy of a duplicated
        pair won depends on it)."""
        import torch
        _req(argmax, torch.int32, "argmax", self.device)
        _req(grad, torch.float32, "grad", self.device)
        if grad.dim() != 2 or grad.shape[0] != self.K or tuple(argmax.shape) != tuple(grad.shape):
            raise ValueError("argmax and grad must both be [M, N] with M the rows of A")
        N = grad.shape[1]
        if B is not None:
            _req(B, torch.float32, "B", self.device)
            if tuple(B.shape) != (self.M, N):
                raise ValueError("B must be [K, N] with K the columns of A")
        elif self.val is not None:
            raise ValueError("a weighted A needs the forward's B for the max backward")
        if out is None:
            out = torch.empty((self.M, N), dtype=torch.float32, device=self.device)
        else:
            _req(out, torch.float32, "out", self.device)
            if tuple(out.shape) != (self.M, N):
                raise ValueError("out has the wrong shape")
        with torch.cuda.device(self.device):
            spmm_maxpool_backward(self.plan, self.col.data_ptr(),
                                  None if self.val is None else self.val.data_ptr(),
                                  None if B is None else B.data_ptr(),
                                  argmax.data_ptr(), grad.data_ptr(), N, out.data_ptr(), stream)
        return out

    def backward(self, grad, reduce: str = "sum", argmax=None, B=None):
        """Gradient with respect to B of ``self.reduce(B, reduce)`` given dC.
        The max needs the forward's argmax and, for a weighted A, its B. The
        transposes are built on first use and kept."""
        if reduce not in REDUCE:
            raise ValueError(f"unknown reduce {reduce!r}")
        if reduce == "mean":
            if self._tmean is None:
                self._tmean = self.transpose(scale_mean=True)
            return self._tmean.reduce(grad, "sum")
        if self._t is None:
            self._t = self.transpose()
        if reduce == "sum":
            return self._t.reduce(grad, "sum")
        if argmax is None:
            raise ValueError("the max backward needs the forward's argmax")
        return self._t.maxpool_backward(argmax, grad, B=B)

    def close(self) -> None:
        for t in (getattr(self, "_t", None), getattr(self, "_tmean", None)):
            if t is not None:
                t.close()
        self._t = self._tmean = None
        if self._plan is not None:
            spmm_plan_destroy(self._plan)
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spmm(rowptr, col, val, mat, reduce: str = "sum"):
    """One-shot product (builds and frees a plan); dispatch by reduce name."""
    adj = SparseAdj(rowptr, col, val, num_cols=mat.shape[0], validate=False)
    try:
        return adj.reduce(mat, reduce)
    finally:
        import torch
        torch.cuda.current_stream(adj.device).synchronize()
        adj.close()


def spmm_sum(rowptr, col, val, mat):
    return spmm(rowptr, col, val, mat, "sum")


def spmm_mean(rowptr, col, val, mat):
    return spmm(rowptr, col, val, mat, "mean")


def spmm_max(rowptr, col, val, mat):
    return spmm(rowptr, col, val, mat, "max")
