// WINDOW family, host side: launch shape (shared-memory layout and pipeline
// depth), the tensor map of B for column-slice rings, and dispatch. The kernel
// is in window.cuh.
#include <cstring>

#include <cudaTypedefs.h>

#include "window.cuh"

namespace spmm {

// ---------------------------------------------------------------- host side
// Shared-memory layout for S pipeline stages (see WinShape).
static void window_layout(WinShape &w, bool has_val, int S) {
    w.S = S;
    w.cap = S * w.R + 2 * w.W;
    w.pow2 = 0;
    int off = 2 * kWinMaxStages * 8;
    w.off_meta = off;
    off += kWinMaxStages * kWinMetaInts * 4;
    off = (off + 15) & ~15;
    w.off_rp = off;
    off += S * w.Rp * 4;
    off = (off + 15) & ~15;
    w.off_col = off;
    off += S * w.ecap * 4;
    w.off_val = off;
    if (has_val) off += S * w.ecap * 4;
    off = (off + 127) & ~127;
    w.off_ring = off;
    w.smem_bytes = off + w.cap * w.cw * 4 + 128;   // + slack to align the base to 128
}

bool window_shape(int64_t M, int64_t K, int64_t N, double dbar, int64_t W, bool has_val,
                  int lanes, int chunks, int rows_per_group, WinShape *o) {
    (void)M; (void)K;
    // the (L, Q) shapes the kernel is instantiated for
    const bool shape_ok = (lanes == 2 && chunks == 1) || (lanes == 4 && chunks == 1) ||
                          (chunks == 2 && (lanes == 2 || lanes == 4 || lanes == 8 || lanes == 16));
    if (!shape_ok || W < 0 || N <= 0) return false;
    if (rows_per_group < 1 || rows_per_group > 2) return false;
    WinShape w{};
    // one or two rows per lane group (two keep more gathers in flight; one keeps
    // the staged entries of high-degree tiles within a stage)
    w.L = lanes;
    w.Q = chunks;
    w.R = rows_per_group * kWinConsumerWarps * kWarp / lanes;
    w.cw = 4 * lanes * chunks;
    // a column slice of B comes by 2-D tensor copies of R-row boxes: W and cap
    // are then multiples of R so that boxes start on a multiple of R and never
    // wrap around the ring
    w.tmap = (w.cw < N) ? 1 : 0;
    w.W = (int)(w.tmap ? (W + w.R - 1) / w.R * w.R : W);
    w.Rp = (w.R + 1 + 3) & ~3;
    int64_t ecap = (int64_t)(w.R * dbar * 1.25) + 64;
    ecap = std::min<int64_t>(4096, std::max<int64_t>(256, (ecap + 3) & ~3));
    w.ecap = (int)ecap;
    // Pipeline depth: one CTA per SM (the consumer warps need more than half of
    // an SM's registers), with as many stages (3 to 8) as shared memory holds.
    int S = 0;
    for (int s = kWinMaxStages; s >= 3 && !S; --s) {
        window_layout(w, has_val, s);
        if (w.smem_bytes <= kWindowSmemBudget) S = s;
    }
    if (!S) S = 3;                                   // too large: the caller rejects it
    window_layout(w, has_val, S);
    w.ctas_per_sm = 1;
    // a power-of-two ring turns the slot of row j into j & (cap - 1)
    int cap2 = 1;
    while (cap2 < w.cap) cap2 <<= 1;
    const int64_t pow2_bytes = (int64_t)w.smem_bytes + (int64_t)(cap2 - w.cap) * w.cw * 4;
    if (pow2_bytes <= kWindowSmemBudget) {
        w.cap = cap2;
        w.pow2 = 1;
        w.smem_bytes = (int)pow2_bytes;
    }
    *o = w;
    return true;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encode_bmap(const RunArgs &a, const WinShape &w, CUtensorMap *map) {
    std::memset(map, 0, sizeof(*map));
    if (!w.tmap) return cudaSuccess;
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
    const cuuint32_t box[2] = {(cuuint32_t)w.cw, (cuuint32_t)w.R};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.B), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_window(const RunArgs &a, const WinShape &w, int reduce, bool has_val, bool check,
                          int grid_x, int tiles, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = encode_bmap(a, w, &map);
    if (e != cudaSuccess) return e;
    switch (reduce) {
        case SPMM_SUM:
            return launch_window_red<SPMM_SUM>(a, w, map, has_val, check, grid_x, tiles, s);
        case SPMM_MEAN:
            return launch_window_red<SPMM_MEAN>(a, w, map, has_val, check, grid_x, tiles, s);
        case SPMM_MAX:
            return launch_window_red<SPMM_MAX>(a, w, map, has_val, check, grid_x, tiles, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace spmm
