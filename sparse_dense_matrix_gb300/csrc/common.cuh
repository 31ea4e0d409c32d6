// Shared definitions of the CUDA library: the plan, the per-launch argument
// block, load/store helpers with cache hints, and the reduction operators.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <climits>

#include "spmm.h"

namespace spmm {

constexpr int kWarp = 32;
constexpr int kMaxTilesY = 65535;
constexpr int kBlockRows = 256;     // diagonal block of the BLOCK (tensor-core) family
// SEGMENT family: merge-path items (stored entries + row ends) per tile, and
// warps per CTA. 544 = 17 * 32, so that the G lane groups of a warp, whose
// slices start 544 / G items apart, read different shared-memory banks when a
// tile lies inside one long row.
#ifndef SPMM_SEG_ITEMS
#define SPMM_SEG_ITEMS 544
#endif
#ifndef SPMM_SEG_WARPS
#define SPMM_SEG_WARPS 16
#endif
constexpr int kSegItems = SPMM_SEG_ITEMS;
constexpr int kSegWarps = SPMM_SEG_WARPS;

// Everything a plan owns. Host-side object; the pointers are device memory.
struct Plan {
    int device = 0;
    int num_sms = 0;
    int64_t M = 0, K = 0, nnz = 0;
    int64_t d_max = 0, n_empty = 0;
    double dbar = 0.0, cv = 0.0;

    int32_t *rowptr = nullptr;       // plan copy of rowptr [M+1], then kRowptrPad copies of rowptr[M]

    // A row-range plan (spmm_plan_create_range) covers rows [row0, row0 + M)
    // of a larger matrix: its rowptr copy is rebased to start at 0, and the
    // caller's full col/val arrays are read from entry col_base = rowptr[row0].
    int64_t row0 = 0, col_base = 0;

    // heavy rows (d > t_split): ids ascending, chunk table (row, begin) per
    // chunk of `chunk` entries, first chunk of each heavy row (prefix, n_heavy+1)
    int64_t t_split = 0, t_split_default = 0;
    int64_t chunk = 0;
    int64_t n_heavy = 0, n_chunks = 0;
    int32_t *heavy_rows = nullptr;
    int32_t *heavy_chunk0 = nullptr;
    int2 *chunks = nullptr;

    // workspace for chunk partials: [n_chunks][N] fp32 (+ int32 for max)
    void *work = nullptr;
    size_t work_bytes = 0;

    // SEGMENT family: merge-path coordinates (rows ended, entries consumed)
    // of the start of every tile of kSegItems items, [seg_n_tiles + 1]
    int2 *seg_tiles = nullptr;
    int64_t seg_n_tiles = 0;

    // BLOCK family, prepared once per plan (block_prepare): every 128-row
    // tile's diagonal block densified and split into TF32 hi/lo operand
    // pieces, and a compact CSR of the entries outside the diagonal blocks.
    // bk_flavor: -1 not prepared, 0 unweighted A, 1 weighted A.
    void *bk_tiles = nullptr;
    int32_t *bk_off_rowptr = nullptr, *bk_off_col = nullptr;
    float *bk_off_val = nullptr;
    int64_t bk_n_off = 0, bk_bytes = 0;
    int bk_flavor = -1;

    // GATHER family, built at its first run (gather_prepare): the row id of
    // every stored entry, [nnz]
    int32_t *ga_rid = nullptr;
    int64_t ga_bytes = 0;

    int32_t *err = nullptr;          // device error words, see kErr*
    int family_override = SPMM_FAMILY_AUTO;

    // column spread |col - row| measured by spmm_plan_validate_cols:
    // spread_hist[b] counts entries with ceil(log2(|col - row|)) == b (0 for 0, 1)
    bool spread_known = false;
    int64_t spread_hist[34] = {0};
    int64_t band_w = 0;              // window half-width chosen from the histogram (0: none)
    bool band_all = false;           // every entry has |col - row| <= band_w
    double band_cover = 0.0;         // fraction of entries with |col - row| <= band_w
    int64_t blk_intra = 0;           // entries inside their row's diagonal kBlockRows block
    bool rows_sorted = false;        // every row's columns non-decreasing
};

// Launch shape of the WINDOW family (host-computed; see f_window.cu).
struct WinShape {
    int R;          // rows per tile (two rows per consumer lane group)
    int W;          // window half-width: tile rows [r0, r1) stage B rows [r0 - W, r1 + W)
    int cap;        // ring rows, >= S R + 2W
    int S;          // pipeline stages
    int ecap;       // col/val entries staged per pipeline stage
    int L, Q;       // lanes per row, 4-column chunks per lane
    int cw;         // B columns held per ring row (4 * L * Q)
    int Rp;         // row-pointer slots per stage (R + 1 rounded up to 4)
    int tmap;       // 1: ring rows are a column slice, loaded by 2-D tensor copies
    int pow2;       // 1: cap is a power of two
    int ctas_per_sm;// CTAs that fit on one SM (shared memory)
    int off_meta, off_rp, off_col, off_val, off_ring, smem_bytes;
};
constexpr int kWindowSmemBudget = 227 * 1024;   // per CTA
constexpr int kWindowSmemPerSm = 228 * 1024;    // per SM
constexpr int kRowptrPad = 1024;    // >= the largest row tile + 4

enum { kErrTimeout = 0, kErrBadCol = 1, kErrWords = 4 };

// Arguments of one spmm_run launch (passed by value to the kernels).
struct RunArgs {
    const int32_t *__restrict__ rowptr;
    const int32_t *__restrict__ col;
    const float *__restrict__ val;
    const float *__restrict__ B;
    float *__restrict__ C;
    int32_t *__restrict__ argmax;
    int64_t M;
    int64_t K;
    int32_t nnz4;       // nnz rounded down to a multiple of 4
    int32_t N;          // feature width (columns of B and C)
    int32_t n_vec;      // N / vec
    int32_t t_split;    // light kernels skip rows with more entries than this
    int32_t chunk;      // entries per heavy-row chunk
    int32_t n_chunks, n_heavy;
    const int2 *__restrict__ chunks;          // (row, begin) per chunk
    const int32_t *__restrict__ heavy_rows;   // [n_heavy]
    const int32_t *__restrict__ heavy_chunk0; // [n_heavy + 1]
    float *__restrict__ ws_val;               // [n_chunks][N]
    int32_t *__restrict__ ws_arg;             // [n_chunks][N] (max only)
    int32_t *__restrict__ err;
    const float *__restrict__ bias;           // [N] added to every output row, or NULL
    int32_t act;                              // spmm_activation applied after the bias
    int32_t rows_sorted;                      // columns non-decreasing within every row
    int32_t mean;                             // 1: a SUM kernel finishes the mean (x 1/d)
    int64_t row0;                             // global index of local row 0 (row-range plans);
                                              // only the WINDOW family's column window uses it
    // SEGMENT family
    const int2 *__restrict__ seg_tiles;       // [seg_n_tiles + 1] (rows ended, entries consumed)
    int64_t seg_n_tiles;
    int32_t seg_warps;                        // warps of the grid (each owns a range of tiles)
    float *__restrict__ seg_cval;             // [tiles_y][seg_warps][2][cw] open-row partials
    int32_t *__restrict__ seg_carg;           // same layout, argmax (max only)
    int4 *__restrict__ seg_meta;              // [seg_warps] (head row, head ends, tail row, 0)
    // BLOCK family (the plan's prepared pieces)
    const void *__restrict__ bk_a;
    const int32_t *__restrict__ bk_off_rowptr;
    const int32_t *__restrict__ bk_off_col;
    const float *__restrict__ bk_off_val;
    float *bk_p;                              // [M][N] off-block partial rows (workspace)
    // GATHER family (the plan's per-entry row ids; its open rows use seg_*)
    const int32_t *__restrict__ ga_rid;
};

// Fused epilogue on V consecutive outputs starting at column c: C = act(C + bias).
// A GCN layer is the aggregation SpMM followed by the node update ("Dual-Metric
// Partitioning with Adaptive Kernel Execution for Efficient GCN Acceleration",
// introduction); applying the bias and activation where C is written saves C a
// round trip. The argmax of max is not affected. ReLU is x > 0 ? x : +0, so -0
// and negative values give +0.
template <int V>
__device__ __forceinline__ void epilogue(const RunArgs &a, int64_t c, float (&out)[V]) {
    if (a.bias) {
#pragma unroll
        for (int e = 0; e < V; ++e) out[e] = __fadd_rn(out[e], __ldg(a.bias + c + e));
    }
    if (a.act == SPMM_ACT_RELU) {
#pragma unroll
        for (int e = 0; e < V; ++e) out[e] = out[e] > 0.0f ? out[e] : 0.0f;
    }
}

// --- global loads / stores with cache hints --------------------------------
// Gathered B rows are re-read by other rows: keep them in L1/L2 (ld.global.nc).
// col / val / rowptr are streamed once: evict-first. C is written once: streaming store.

__device__ __forceinline__ int ld_stream(const int32_t *p) { return __ldcs(p); }
__device__ __forceinline__ float ld_stream(const float *p) { return __ldcs(p); }

template <int V> struct VecT;
template <> struct VecT<1> { using type = float; };
template <> struct VecT<4> { using type = float4; };

template <int V>
__device__ __forceinline__ void ld_vec(const float *p, float (&x)[V]) {
    if constexpr (V == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        x[0] = __ldg(p);
    }
}

template <int V>
__device__ __forceinline__ void st_vec(float *p, const float (&x)[V]) {
    if constexpr (V == 4) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    } else {
        __stcs(p, x[0]);
    }
}

template <int V>
__device__ __forceinline__ void st_vec_i(int32_t *p, const int (&x)[V]) {
    if constexpr (V == 4) {
        __stcs(reinterpret_cast<int4 *>(p), make_int4(x[0], x[1], x[2], x[3]));
    } else {
        __stcs(p, x[0]);
    }
}

// --- reductions -------------------------------------------------------------
// sum / mean: fp32 fused multiply-add per entry; the order is fixed by the
// kernel's mapping. max: (value, column) with the total order "larger value,
// then smaller column"; the identity (-inf, INT_MAX) marks "no entry yet".

constexpr int kNoCol = INT_MAX;

// Reciprocal by the PTX rcp.approx.f32 instruction (at most 1 ulp from 1/x);
// the mean is then fl(sum * rcp(d)), a few ulp from the correctly rounded
// quotient, far inside the sum/mean tolerance.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ bool max_better(float y, int jy, float v, int jv) {
    return y > v || (y == v && jy < jv);
}

template <int V, int RED, bool HAS_VAL>
struct Acc {
    float v[V];
    int j[V];   // used by max only

    __device__ __forceinline__ void init() {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            v[e] = (RED == SPMM_MAX) ? -__int_as_float(0x7f800000) : 0.0f;
            j[e] = kNoCol;
        }
    }

    __device__ __forceinline__ void add(float a, int col, const float (&b)[V]) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            if constexpr (RED == SPMM_MAX) {
                const float y = HAS_VAL ? __fmul_rn(a, b[e]) : b[e];
                if (max_better(y, col, v[e], j[e])) { v[e] = y; j[e] = col; }
            } else {
                v[e] = HAS_VAL ? __fmaf_rn(a, b[e], v[e]) : __fadd_rn(v[e], b[e]);
            }
        }
    }

    // combine with the accumulator held by lane (lane ^ offset)
    __device__ __forceinline__ void combine_xor(int offset) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const float ov = __shfl_xor_sync(0xffffffffu, v[e], offset);
            if constexpr (RED == SPMM_MAX) {
                const int oj = __shfl_xor_sync(0xffffffffu, j[e], offset);
                if (max_better(ov, oj, v[e], j[e])) { v[e] = ov; j[e] = oj; }
            } else {
                // both partners compute the same sum (a + b == b + a bit for bit)
                v[e] = __fadd_rn(v[e], ov);
            }
        }
    }

    // final values for a row of d stored entries (mean: one reciprocal of d per
    // row, then a product per element)
    __device__ __forceinline__ void finish(int d, float (&out)[V], int (&arg)[V]) const {
        const float inv_d = (RED == SPMM_MEAN && d > 0) ? rcp_approx((float)d) : 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            if constexpr (RED == SPMM_MAX) {
                const bool none = (j[e] == kNoCol);
                out[e] = none ? 0.0f : v[e];
                arg[e] = none ? -1 : j[e];
            } else if constexpr (RED == SPMM_MEAN) {
                out[e] = __fmul_rn(v[e], inv_d);
                arg[e] = 0;
            } else {
                out[e] = v[e];
                arg[e] = 0;
            }
        }
    }
};

// The mean finished by a SUM kernel (the row-per-warp families run the mean as
// the sum plus this step): fl(S * rcp(d)) as Acc<..., MEAN>::finish, 0 for d = 0.
template <int V>
__device__ __forceinline__ void mean_scale(const RunArgs &a, int d, float (&out)[V]) {
    if (a.mean) {
        const float inv_d = d > 0 ? rcp_approx((float)d) : 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) out[e] = __fmul_rn(out[e], inv_d);
    }
}

// Number of kernels launched by this library (spmm_launch_count).
extern std::atomic<uint64_t> g_launches;
inline void count_launch(uint64_t n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Family launchers (one translation unit each). Return a CUDA error code.
cudaError_t launch_rowgroup(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                            int tiles, cudaStream_t s);
cudaError_t launch_warprow(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                           int tiles, cudaStream_t s);
cudaError_t launch_heavy(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                         int tiles, cudaStream_t s);
cudaError_t launch_coltile(const RunArgs &a, int wpr, int tiles_y, int reduce, bool has_val,
                           bool bulk_ok, cudaStream_t s);
cudaError_t launch_window(const RunArgs &a, const WinShape &w, int reduce, bool has_val, bool check,
                          int grid_x, int tiles, cudaStream_t s);
bool window_shape(int64_t M, int64_t K, int64_t N, double dbar, int64_t W, bool has_val,
                  int lanes, int chunks, int rows_per_group, WinShape *out);
cudaError_t launch_block(const RunArgs &a, int reduce, bool has_val, cudaStream_t s);
// BLOCK preparation from the plan's rowptr and the caller's col/val (synchronous)
cudaError_t block_prepare(Plan *p, const int32_t *col, const float *val, cudaStream_t s);
void block_free(Plan *p);
size_t block_prepared_bytes(int64_t M, int64_t n_off, bool has_val);
// SEGMENT: main kernel (ctas_x x tiles_y CTAs) and the combine of the open rows
cudaError_t launch_segment(const RunArgs &a, int lanes, int chunks, int reduce, bool has_val,
                           int tiles_y, cudaStream_t s);
// workspace bytes of the SEGMENT family's open-row partials for a launch
size_t segment_workspace(int64_t seg_warps, int64_t tiles_y, int lanes, int chunks, int reduce);
// warps of a SEGMENT launch on `num_sms` SMs with `tiles_y` column tiles
int64_t segment_warps(int64_t n_tiles, int num_sms, int64_t tiles_y);
// GATHER: column tile (256 or 128 columns, 0 if N fits neither), CTAs of a
// launch, open-row workspace bytes, the per-entry row ids (once per plan),
// and the launch of the main kernel plus the open-row combine
int gather_tile(int64_t N);
int64_t gather_ctas(int64_t nnz, int num_sms, int64_t tiles_y);
size_t gather_workspace(int64_t ctas, int64_t tiles_y, int ct, int reduce);
cudaError_t gather_prepare(Plan *p, cudaStream_t s);
void gather_free(Plan *p);
cudaError_t launch_gather(const RunArgs &a, int reduce, bool has_val, int ctas, int tiles_y,
                          cudaStream_t s);
// STREAM: lanes per range (16 or 32; 0 when N % 4 != 0 or N <= 32), ranges of
// a launch, open-row workspace bytes, and the launch of the main kernel plus
// the open-row combine (the per-entry row ids come from gather_prepare)
int stream_lanes(int64_t N);
int64_t stream_ranges(int64_t nnz, int num_sms, int lanes, int64_t tiles_y);
size_t stream_workspace(int64_t ranges, int64_t tiles_y, int lanes, int reduce);
cudaError_t launch_stream(const RunArgs &a, int reduce, bool has_val, int lanes, int64_t ranges,
                          int tiles_y, cudaStream_t s);
// grow a plan's workspace to at least `need` bytes (cudaMalloc; synchronous)
spmm_status plan_ensure_workspace(Plan *p, size_t need);

}  // namespace spmm
