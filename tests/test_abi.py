"""The C ABI without a GPU: the library loads, exports every declared symbol,
rejects bad arguments on the host, and its router is a pure function."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sdm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_dense_matrix_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "spmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spmm_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("spmm_plan_create", "spmm_run", "spmm_plan_describe", "spmm_plan_destroy",
                 "spmm_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(sdm):
    lib = ctypes.CDLL(os.path.join(ROOT, "sparse_dense_matrix_gb300", "libspmm.so"))
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(sdm):
    for code in range(7):
        assert sdm.spmm_status_string(code)
    assert sdm.spmm_status_string(0) == "ok"
    assert "unknown" in sdm.spmm_status_string(99)


def test_host_argument_checks(sdm):
    lib = sdm.lib
    out = ctypes.c_void_p(123)
    assert lib.spmm_plan_create(None, 10, 10, None, ctypes.byref(out)) == 1
    assert out.value is None                      # cleared on error
    assert lib.spmm_plan_create(ctypes.c_void_p(16), -1, 10, None, ctypes.byref(out)) == 1
    assert lib.spmm_plan_create(ctypes.c_void_p(16), 10, 10, None, None) == 1
    assert lib.spmm_plan_create(ctypes.c_void_p(16), 1 << 31, 10, None, ctypes.byref(out)) == 5
    assert lib.spmm_run(None, None, None, None, 4, 0, None, None, None) == 1
    assert lib.spmm_plan_reserve(None, 4, 0) == 1
    assert lib.spmm_plan_validate_cols(None, None, None) == 1
    assert lib.spmm_plan_sync(None, None) == 1
    assert lib.spmm_plan_prepare_blocks(None, None, None, None) == 1
    info = sdm.PlanInfo()
    assert lib.spmm_plan_describe(None, 4, 0, ctypes.byref(info)) == 1
    assert lib.spmm_plan_set_family(None, 0, 0) == 1
    assert lib.spmm_plan_destroy(None) == 0
    assert lib.spmm_transpose(None, None, None, 0, None, None, None, None) == 1
    assert lib.spmm_check_wait_timeout(None, 1000, None) == 1
    assert lib.spmm_check_wait_timeout(ctypes.c_void_p(16), 0, None) == 1
    assert lib.spmm_maxpool_backward(None, None, None, None, None, None, 4, None, None) == 1
    assert lib.spmm_maxpool_backward(ctypes.c_void_p(16), None, None, None, None, None, -1, None,
                                     None) == 1
    assert lib.spmm_route(ctypes.byref(info), 4, 7, 1, 152, -1, ctypes.byref(info)) == 1
    assert lib.spmm_route(ctypes.byref(info), -4, 0, 1, 152, -1, ctypes.byref(info)) == 1
    assert lib.spmm_route(ctypes.byref(info), 4, 0, 1, 152, 9, ctypes.byref(info)) == 1
    assert lib.spmm_plan_create_range(None, 0, 4, 10, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert lib.spmm_plan_create_range(ctypes.c_void_p(16), 5, 4, 10, None, ctypes.byref(out)) == 1
    assert lib.spmm_plan_create_range(ctypes.c_void_p(16), -1, 4, 10, None, ctypes.byref(out)) == 1
    assert lib.spmm_plan_create_range(ctypes.c_void_p(16), 0, 4, 10, None, None) == 1
    assert lib.spmm_plan_create_range(ctypes.c_void_p(16), 0, 1 << 31, 10, None,
                                      ctypes.byref(out)) == 5
    b = (ctypes.c_int64 * 3)()
    assert lib.spmm_partition_rows(None, 4, 2, 1, b) == 1


def test_plan_create_without_a_gpu_reports_cuda_error(sdm):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful on a host without a GPU")
    out = ctypes.c_void_p()
    # never dereferenced: the device query fails first
    assert sdm.lib.spmm_plan_create(ctypes.c_void_p(4096), 10, 10, None, ctypes.byref(out)) == 4


def _desc(M=1 << 20, nnz=10 << 20, cv=0.0, n_heavy=0, n_chunks=0, t_split=512):
    return dict(M=M, K=M, nnz=nnz, dbar=nnz / M, cv=cv, d_max=10, n_empty=0,
                t_split=t_split, chunk=t_split // 2, n_heavy=n_heavy, n_chunks=n_chunks,
                seg_tiles=(M + nnz + 543) // 544)


def test_router_rules(sdm):
    r = sdm.spmm_route(_desc(cv=0.0), 16, 0)
    assert (r["family_name"], r["vec"], r["lanes"], r["rows_per_warp"], r["col_tiles"]) == \
        ("rowgroup", 4, 4, 8, 1)
    r = sdm.spmm_route(_desc(cv=0.0), 64, 1)
    assert (r["family_name"], r["lanes"], r["rows_per_warp"]) == ("rowgroup", 16, 2)
    r = sdm.spmm_route(_desc(cv=9.2), 64, 0)
    assert (r["family_name"], r["lanes"], r["rows_per_warp"]) == ("warprow", 16, 1)
    r = sdm.spmm_route(_desc(cv=0.1), 512, 0)                 # wide N: column tiles
    assert (r["family_name"], r["vec"], r["lanes"], r["col_tiles"]) == ("warprow", 4, 32, 4)
    r = sdm.spmm_route(_desc(cv=0.1), 512, 0, aligned=0)      # no 128-bit vectors
    assert (r["family_name"], r["vec"], r["col_tiles"]) == ("warprow", 1, 16)
    r = sdm.spmm_route(_desc(cv=0.1), 64, 0, family=sdm.FAMILY["coltile"])
    assert (r["family_name"], r["lanes"], r["col_tiles"]) == ("coltile", 32, 1)
    r = sdm.spmm_route(_desc(cv=0.0), 16, 0, aligned=False)    # scalar path
    assert (r["vec"], r["lanes"], r["rows_per_warp"]) == (1, 16, 2)
    r = sdm.spmm_route(_desc(cv=0.0), 17, 0)                   # N % 4 != 0
    assert (r["vec"], r["lanes"], r["col_tiles"]) == (1, 32, 1)
    r = sdm.spmm_route(_desc(cv=0.0), 33, 0)
    assert (r["family_name"], r["vec"], r["col_tiles"]) == ("warprow", 1, 2)
    assert sdm.spmm_route(_desc(cv=0.0), 36, 0)["family_name"] == "rowgroup"
    r = sdm.spmm_route(_desc(cv=0.0), 128, 0)                  # 32 lanes: a warp per row
    assert (r["family_name"], r["lanes"], r["rows_per_warp"]) == ("warprow", 32, 1)
    r = sdm.spmm_route(_desc(cv=0.0), 1, 2)
    assert (r["vec"], r["lanes"], r["rows_per_warp"]) == (1, 2, 16)
    r = sdm.spmm_route(_desc(cv=0.0), 16, 0, family=sdm.FAMILY["warprow"])
    assert r["family_name"] == "warprow"


def test_router_segment_rule(sdm):
    """Skewed degrees at N <= 32 with 128-bit vectors and aligned col/val go to
    the merge-path SEGMENT family: two launches, no split-row launches, a
    workspace of two partial rows per warp (+ a 16-byte record per warp)."""
    d = _desc(M=1 << 22, nnz=104_839_949, cv=20.6, n_heavy=9000, n_chunks=90000)
    for N in (4, 8, 16, 32):
        r = sdm.spmm_route(d, N, 0, aligned=3)
        assert r["family_name"] == "segment", N
        assert r["launches"] == 2 and r["seg_warps"] == 152 * 16 and r["col_tiles"] == 1
    r = sdm.spmm_route(d, 16, 0, aligned=3)
    assert r["workspace_bytes"] == 152 * 16 * 16 + 152 * 16 * 2 * 16 * 4
    r = sdm.spmm_route(d, 16, 2, aligned=3)                    # + argmax partials
    assert r["workspace_bytes"] == 152 * 16 * 16 + 2 * 152 * 16 * 2 * 16 * 4
    assert sdm.spmm_route(d, 16, 0, aligned=1)["family_name"] == "warprow"   # col/val unaligned
    assert sdm.spmm_route(d, 64, 0, aligned=3)["family_name"] == "warprow"   # wider N
    assert sdm.spmm_route(d, 18, 0, aligned=3)["family_name"] == "warprow"   # no 128-bit vectors
    assert sdm.spmm_route(_desc(cv=0.5), 16, 0, aligned=3)["family_name"] == "rowgroup"
    pin = sdm.FAMILY["segment"]
    r = sdm.spmm_route(d, 1000, 0, aligned=3, family=pin)      # two chunks per lane, 4 tiles
    assert (r["family_name"], r["lanes"], r["seg_chunks"], r["col_tiles"]) == ("segment", 32, 2, 4)
    assert r["seg_warps"] == 152 // 4 * 16
    assert sdm.spmm_route(d, 6, 0, aligned=3, family=pin)["family_name"] == "warprow"


def test_router_gather_rule(sdm):
    """Pinned GATHER: column tiles of 256 (else 128) columns that N fills
    exactly, two CTAs per SM shared among the tiles but never more CTAs than
    entries, two launches, no split-row launches, a workspace of two partial
    rows per CTA (+ a 16-byte record per CTA, rounded to 256 bytes)."""
    pin = sdm.FAMILY["gather"]
    d = _desc(M=1 << 22, nnz=104_839_949, cv=20.6, n_heavy=9000, n_chunks=90000)
    r = sdm.spmm_route(d, 256, 0, aligned=3, family=pin)
    assert (r["family_name"], r["col_tiles"], r["gather_ctas"], r["launches"]) == \
        ("gather", 1, 304, 2)
    assert r["workspace_bytes"] == 304 * 16 + 304 * 2 * 256 * 4
    r = sdm.spmm_route(d, 256, 2, aligned=1, family=pin)       # + argmax partials
    assert r["workspace_bytes"] == 304 * 16 + 2 * 304 * 2 * 256 * 4
    r = sdm.spmm_route(d, 384, 0, aligned=1, family=pin)       # three tiles of 128
    assert (r["family_name"], r["col_tiles"], r["gather_ctas"]) == ("gather", 3, 101)
    assert r["workspace_bytes"] == (101 * 16 + 255) // 256 * 256 + 3 * 101 * 2 * 128 * 4
    r = sdm.spmm_route(d, 512, 0, aligned=1, family=pin)       # two tiles of 256
    assert (r["col_tiles"], r["gather_ctas"]) == (2, 152)
    r = sdm.spmm_route(_desc(M=5, nnz=6), 128, 0, aligned=1, family=pin)
    assert (r["family_name"], r["gather_ctas"]) == ("gather", 6)   # one CTA per entry
    for N, aligned, dd in ((64, 3, d), (130, 3, d), (256, 2, d), (256, 3, _desc(nnz=0))):
        assert sdm.spmm_route(dd, N, 0, aligned=aligned, family=pin)["family_name"] != "gather"


def test_router_stream_rule(sdm):
    """Pinned STREAM: 16 lanes per range up to N = 64, else 32 lanes per
    128-column tile; two waves of 4 x 256-thread blocks per SM shared among
    the tiles, 32 / lanes ranges per warp, at least 16 entries a range; two
    launches, no split-row launches, a workspace of two partial rows per range
    (+ a 16-byte record per range, rounded to 256 bytes)."""
    pin = sdm.FAMILY["stream"]
    d = _desc(M=1 << 22, nnz=104_839_949, cv=20.6, n_heavy=9000, n_chunks=90000)
    r = sdm.spmm_route(d, 64, 0, aligned=3, family=pin)
    assert (r["family_name"], r["lanes"], r["col_tiles"], r["stream_ranges"], r["launches"]) == \
        ("stream", 16, 1, 19456, 2)
    assert r["workspace_bytes"] == 19456 * 16 + 19456 * 2 * 64 * 4
    r = sdm.spmm_route(d, 256, 2, aligned=1, family=pin)       # + argmax partials
    assert (r["lanes"], r["col_tiles"], r["stream_ranges"]) == (32, 2, 4864)
    assert r["workspace_bytes"] == 4864 * 16 + 2 * 2 * 4864 * 2 * 128 * 4
    r = sdm.spmm_route(d, 48, 0, aligned=1, family=pin)        # 12 of 16 lanes active
    assert (r["family_name"], r["lanes"], r["col_tiles"]) == ("stream", 16, 1)
    r = sdm.spmm_route(_desc(M=5, nnz=6), 128, 0, aligned=1, family=pin)
    assert (r["family_name"], r["stream_ranges"]) == ("stream", 1)
    for N, aligned, dd in ((32, 3, d), (66, 3, d), (256, 2, d), (256, 3, _desc(nnz=0))):
        assert sdm.spmm_route(dd, N, 0, aligned=aligned, family=pin)["family_name"] != "stream"


def test_router_split_launches_and_workspace(sdm):
    r = sdm.spmm_route(_desc(cv=9.0, n_heavy=3, n_chunks=40), 64, 0)
    assert r["launches"] == 3 and r["workspace_bytes"] == 40 * 64 * 4
    r = sdm.spmm_route(_desc(cv=9.0, n_heavy=3, n_chunks=40), 64, 2)
    assert r["workspace_bytes"] == 2 * 40 * 64 * 4             # values + argmax partials
    r = sdm.spmm_route(_desc(), 64, 0)
    assert r["launches"] == 1 and r["workspace_bytes"] == 0
    r = sdm.spmm_route(_desc(), 0, 0)
    assert r["launches"] == 0


def test_default_split_threshold(sdm):
    assert sdm.spmm_default_t_split(2048, 16384, 152) == 256
    assert sdm.spmm_default_t_split(1 << 22, 104_839_949, 152) == 512
    assert sdm.spmm_default_t_split(1 << 20, 128 * 152 * 300, 152) == 300
    assert sdm.spmm_default_t_split(10, 10, 0) == 256


def test_tensor_api_refuses_cpu_tensors(sdm):
    torch = pytest.importorskip("torch")
    rp = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        sdm.SparseAdj(rp, torch.zeros(0, dtype=torch.int32))


def test_router_window_rule(sdm):
    knn = dict(_desc(cv=0.0), band_w=512, band_cover=0.999)
    r = sdm.spmm_route(knn, 16, 0)
    assert (r["family_name"], r["lanes"], r["window_chunks"], r["col_tiles"], r["window_rows"]) == \
        ("window", 4, 1, 1, 256)
    assert 0 < r["window_smem"] <= 227 * 1024 and r["window_ctas"] == 152
    r = sdm.spmm_route(knn, 64, 1)
    assert (r["family_name"], r["lanes"], r["window_chunks"], r["col_tiles"], r["window_ctas"]) == \
        ("window", 4, 2, 2, 76)
    r = sdm.spmm_route(knn, 8, 0)
    assert (r["family_name"], r["lanes"], r["window_chunks"], r["col_tiles"]) == ("window", 2, 1, 1)
    community = dict(_desc(M=65536, nnz=3668321, cv=0.1), band_w=256, band_cover=0.91)
    assert sdm.spmm_route(community, 128, 0)["family_name"] != "window"          # 9% outside W
    dense_band = dict(community, band_cover=0.99)   # 56 entries per row: a tile overflows a stage
    assert sdm.spmm_route(dense_band, 128, 0)["family_name"] != "window"
    assert sdm.spmm_route(dense_band, 512, 0)["family_name"] != "window"         # ring too big
    assert sdm.spmm_route(knn, 64, 0, aligned=1)["family_name"] == "rowgroup"   # col unaligned
    assert sdm.spmm_route(knn, 18, 0)["family_name"] != "window"                 # N % 4 != 0
    assert sdm.spmm_route(_desc(cv=0.0), 16, 0)["family_name"] == "rowgroup"    # spread unknown
    small = dict(_desc(M=4096, nnz=40960, cv=0.0), band_w=512, band_cover=0.99)
    assert sdm.spmm_route(small, 16, 0)["family_name"] == "rowgroup"            # halo too large
    r = sdm.spmm_route(small, 16, 0, family=sdm.FAMILY["window"])
    assert r["family_name"] == "window"                                           # pinned
    wide = dict(_desc(cv=0.0), band_w=4096, band_cover=0.9)
    assert sdm.spmm_route(wide, 512, 0)["family_name"] == "warprow"             # ring too big
    # row-range plans: the tiles must start on whole R-row boxes of B
    assert sdm.spmm_route(dict(knn, row0=1 << 19), 16, 0)["family_name"] == "window"
    assert sdm.spmm_route(dict(knn, row0=1 << 19), 64, 0)["family_name"] == "window"
    assert sdm.spmm_route(dict(knn, row0=1000), 16, 0)["family_name"] == "rowgroup"
    r = sdm.spmm_route(dict(knn, row0=128), 16, 0)          # 256-row tiles do not fit: 128
    assert (r["family_name"], r["window_rows"]) == ("window", 128)
    assert sdm.spmm_route(dict(knn, row0=64), 16, 0)["family_name"] == "rowgroup"


def test_router_block_rule(sdm):
    # community 64k: 256 blocks of 256 rows, 51 of 56 entries per row inside the
    # block (91%, block density 0.2): routed to BLOCK for sum and mean
    com = dict(_desc(M=65536, nnz=3668321, cv=0.1), band_w=256, band_cover=0.91,
               rows_sorted=1, blk_intra=3342000)
    assert sdm.spmm_route(com, 128, 0)["family_name"] == "block"
    assert sdm.spmm_route(com, 512, 1)["family_name"] == "block"
    assert sdm.spmm_route(com, 128, 2)["family_name"] != "block"                # max
    assert sdm.spmm_route(dict(com, blk_intra=0), 128, 0)["family_name"] != "block"  # unknown
    assert sdm.spmm_route(dict(com, blk_intra=3000000), 128, 0)["family_name"] != "block"  # 82%
    sparse_blocks = dict(_desc(M=65536, nnz=500000, cv=0.1), blk_intra=480000)   # 2.9% dense
    assert sdm.spmm_route(sparse_blocks, 128, 0)["family_name"] != "block"
    assert sdm.spmm_route(com, 128, 0, family=sdm.FAMILY["warprow"])["family_name"] == "warprow"
    pin = sdm.FAMILY["block"]
    r = sdm.spmm_route(com, 128, 0, family=pin)
    assert (r["family_name"], r["col_tiles"], r["launches"]) == ("block", 1, 1)
    assert sdm.spmm_route(com, 512, 1, family=pin)["col_tiles"] == 4            # mean too
    assert sdm.spmm_route(com, 128, 2, family=pin)["family_name"] != "block"   # max
    assert sdm.spmm_route(com, 40, 0, family=pin)["family_name"] != "block"    # N % 16
    r = sdm.spmm_route(com, 128, 0, aligned=2, family=pin)
    assert r["family_name"] != "block"                                          # unaligned B/C
    r = sdm.spmm_route(dict(com, rows_sorted=0), 128, 0, family=pin)
    assert r["family_name"] == "block"                                          # any row order
    r = sdm.spmm_route(dict(com, row0=256), 128, 0, family=pin)
    assert r["family_name"] == "warprow"                                        # a row range

