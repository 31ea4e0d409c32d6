/*
 * spmm.h -- C ABI of the GB300 CSR SpMM engine (libspmm.so).
 *
 * The engine computes C = A . B for a fixed sparse M x K matrix A in CSR and a
 * dense K x N fp32 matrix B, under a sum, mean or max reduction; max also
 * returns the winning column (argmax). Semantics follow the graph-spmm model
 * card ("API", "Method", "Correctness"): `val == NULL` is an unweighted
 * adjacency, duplicate (row, col) entries are each counted, an empty row gives
 * 0 for sum and mean and (0, -1) for max, and ties of max go to the smallest
 * column. The row-wise CSR traversal is ParamSpMM section 2 ("Background",
 * Algorithm 1); the plan's O(M) degree descriptors are RA-SpMM's (abstract and
 * "routing rules": M, mean degree, degree coefficient of variation).
 *
 * Conventions for every call
 *   - Pointers named "device" are CUDA device pointers of the current device;
 *     the library never dereferences them on the host.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued on it; calls marked "synchronous" also wait
 *     for it to drain before they return.
 *   - Every call returns an spmm_status; no C++ exception crosses the ABI and
 *     no device code traps. Argument checks happen on the host before any CUDA
 *     call, so an invalid-argument status is returned even on a machine
 *     without a GPU.
 *   - The caller owns all tensors (rowptr, col, val, B, C, argmax). The plan
 *     owns its own copy of rowptr, its heavy-row tables and its workspace.
 *   - A plan may be used by one stream at a time (it owns one workspace).
 *   - Results are bitwise reproducible run to run: no floating-point atomics,
 *     every reduction order is a pure function of the plan and N.
 */
#ifndef GB300_SPMM_H
#define GB300_SPMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPMM_OK = 0,
    SPMM_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, unknown enum value      */
    SPMM_ERR_INVALID_INPUT = 2, /* rowptr not a CSR row-pointer array; col out of range */
    SPMM_ERR_OOM = 3,           /* device or host allocation failed                     */
    SPMM_ERR_CUDA = 4,          /* a CUDA runtime call failed (no device, launch error)  */
    SPMM_ERR_UNSUPPORTED = 5,   /* size beyond the int32 index range                     */
    SPMM_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up (see spmm_plan_sync) */
} spmm_status;

/* graph-spmm model card, "API": spmm_sum / spmm_mean / spmm_max. */
typedef enum { SPMM_SUM = 0, SPMM_MEAN = 1, SPMM_MAX = 2 } spmm_reduce;

/* Activation of the fused epilogue (spmm_run_ex). */
typedef enum { SPMM_ACT_NONE = 0, SPMM_ACT_RELU = 1 } spmm_activation;

/* Kernel families the router chooses among (RA-SpMM "kernel portfolio" and
 * "routing rules": the family is picked from the descriptors and N). */
typedef enum {
    SPMM_FAMILY_AUTO = -1,     /* let the router decide                                  */
    SPMM_FAMILY_ROWGROUP = 0,  /* several rows per warp, L lanes per row (uniform degree) */
    SPMM_FAMILY_WARPROW = 1,   /* one warp per row, lane groups split the row's entries   */
    SPMM_FAMILY_COLTILE = 2,   /* a CTA per row block, warps own 128-column tiles, col/val
                                  staged in shared memory (wide N)                         */
    SPMM_FAMILY_WINDOW = 3,    /* persistent CTAs over contiguous row ranges; the B rows of a
                                  sliding window [r0 - W, r1 + W) are streamed into shared
                                  memory by bulk copies (column-locality graphs)           */
    SPMM_FAMILY_BLOCK = 4,     /* block-diagonal graphs: each 128-row tile's 256-column
                                  diagonal block, densified and split into TF32 hi + lo once
                                  per plan (spmm_plan_prepare_blocks), is multiplied on the
                                  tensor cores (fp32 accumulation); the entries outside the
                                  block, also prepared, are added by the same CTA. Sum and
                                  mean, N % 16 == 0, aligned B and C, a plan of whole rows
                                  (not a row range)                                          */
    SPMM_FAMILY_SEGMENT = 5,   /* skewed graphs without column locality: the CSR traversal is
                                  cut into equal merge-path tiles of entries plus row ends
                                  (ParamSpMM section 3.2, nonzero-split balancing); each warp
                                  streams its tiles' rowptr/col/val into shared memory with
                                  bulk copies and reduces them in lane-group slices, rows
                                  open across tiles carried in registers, the few rows open
                                  at the ends of a warp's range combined by a second launch.
                                  N % 4 == 0, 16-byte aligned B, C, argmax, col and val;
                                  long rows need no separate split                          */
    SPMM_FAMILY_GATHER = 6,    /* skewed graphs at wide N: equal contiguous entry ranges, one
                                  per CTA; a producer warp streams the range's col/val and
                                  the plan's per-entry row ids and has the tensor-copy engine
                                  gather the entries' B rows (tile::gather4, four rows per
                                  copy) into a shared-memory ring; four consumer warps own a
                                  quarter of the column tile each and walk the entries in
                                  CSR order. The rows open at the ends of a CTA's range are
                                  combined by a second launch. N % 128 == 0, 16-byte aligned
                                  B, C and argmax; the row ids (4 bytes per entry) are built
                                  at the plan's first GATHER run                            */
    SPMM_FAMILY_STREAM = 7     /* skewed graphs at N > 32: the entries as one stream cut into
                                  equal contiguous ranges, one per lane group (16 lanes for
                                  N <= 64, else 32 per 128-column tile); each group loads the
                                  columns, values and per-entry row ids of its next 32
                                  entries while gathering the current ones, and finishes a
                                  row when the row id changes. The rows open at the ends of
                                  a range are combined by a second launch. N % 4 == 0,
                                  16-byte aligned B, C and argmax; shares GATHER's row ids */
} spmm_family;

typedef struct spmm_plan_s *spmm_plan_t;

/* Descriptors and routing decision, filled by spmm_plan_describe / spmm_route. */
typedef struct {
    /* O(M) descriptors of the row-degree distribution */
    int64_t M, K, nnz;
    int64_t d_max;          /* largest row degree                                    */
    int64_t n_empty;        /* rows with no entry                                    */
    double dbar;            /* nnz / M (0 when M == 0)                               */
    double cv;              /* std(d) / mean(d) over all M rows, divisor M (0 if nnz==0) */
    /* heavy-row split (rows longer than t_split are cut into chunks of `chunk` entries,
     * reduced per chunk, then combined in chunk order by a second launch) */
    int64_t t_split;
    int64_t chunk;
    int64_t n_heavy;
    int64_t n_chunks;
    /* launch shape for the queried (N, reduce) */
    int64_t N;
    int32_t reduce;
    int32_t family;         /* spmm_family actually used                             */
    int32_t vec;            /* columns per lane load: 4 (128-bit) or 1               */
    int32_t lanes;          /* lanes that share one entry (one per vec of columns)   */
    int32_t rows_per_warp;  /* rows one warp owns (ROWGROUP), else 1                 */
    int32_t col_tiles;      /* column tiles (grid dimension y): lanes*vec columns each, 
                               WINDOW: 4*lanes*window_chunks columns each             */
    int32_t launches;       /* kernel launches one spmm_run makes                    */
    int32_t num_sms;        /* SM count the routing assumed                          */
    int64_t workspace_bytes;/* device scratch spmm_run needs for this (N, reduce)    */
    /* column locality, known after spmm_plan_validate_cols (0 before) */
    int64_t band_w;         /* smallest power of two W with >= 85% of entries at |col - row| <= W,
                               0 if none up to 4096                                       */
    double band_cover;      /* fraction of entries with |col - row| <= band_w           */
    int32_t window_rows;    /* WINDOW family: rows per tile (0 for other families)      */
    int32_t window_ctas;    /* WINDOW family: CTAs per column tile                      */
    int64_t window_smem;    /* WINDOW family: dynamic shared memory per CTA, bytes      */
    int32_t window_chunks;  /* WINDOW family: 4-column chunks per lane (cw = 4 lanes x chunks) */
    /* block structure, known after spmm_plan_validate_cols (0 before) */
    int32_t rows_sorted;    /* 1 if every row's columns are non-decreasing             */
    int64_t blk_intra;      /* entries with col / 256 == row / 256 (diagonal blocks)     */
    /* row-range plans (spmm_plan_create_range): global index of the plan's row 0 */
    int64_t row0;
    /* SEGMENT family: merge-path tiles of the plan (descriptor), and for the
       queried (N, reduce) the warps of the grid and the four-column chunks per lane */
    int64_t seg_tiles;
    int32_t seg_warps;
    int32_t seg_chunks;
    /* BLOCK family: device bytes of the plan's prepared diagonal blocks and
       off-block entries (0 until prepared) */
    int64_t block_bytes;
    /* GATHER family: device bytes of the plan's per-entry row ids (0 until its
       first run), and for the queried (N, reduce) the CTAs per column tile */
    int64_t gather_bytes;
    int32_t gather_ctas;
    /* STREAM family: for the queried (N, reduce) the entry ranges of the grid */
    int32_t stream_ranges;
} spmm_plan_info;

/*
 * spmm_plan_create -- build the reusable plan for one sparsity pattern.
 *   rowptr : device, int32 [M+1], rowptr[0] == 0, non-decreasing. Copied into
 *            plan-owned memory; the caller may free it after the call returns.
 *   M, K   : rows and columns of A (M >= 0, K >= 0, both < 2^31).
 *   stream : work is enqueued here. Synchronous.
 *   out    : receives the plan (left NULL on error).
 * Computes, in one pass over rowptr, the degree descriptors (M, nnz, mean
 * degree, degree CV, max degree, empty rows) and the list of heavy rows that
 * spmm_run splits across CTAs, and, by a binary search per tile, the SEGMENT
 * family's merge-path tile table (the rows ended and entries consumed at every
 * 544th item of entries plus row ends; 8 bytes per tile). Returns SPMM_ERR_INVALID_INPUT when rowptr[0]
 * != 0 or rowptr decreases anywhere (checked on the device; no trap).
 * (RA-SpMM abstract: descriptors in O(M); graph-spmm model card, "API":
 * SparseAdj is held once and applied many times.)
 */
spmm_status spmm_plan_create(const int32_t *rowptr, int64_t M, int64_t K, void *stream,
                             spmm_plan_t *out);

/*
 * spmm_plan_create_range -- a plan for the contiguous rows [row_begin, row_end)
 * of a larger CSR matrix: one worker's share when rows are split across
 * workers (each row's output depends on that row alone, so the shares need no
 * exchange). Built like spmm_plan_create over those rows.
 *   rowptr    : device (or host), int32 [>= row_end + 1], the WHOLE matrix's
 *               row pointers; entries row_begin .. row_end are copied and
 *               rebased to start at 0. rowptr[0] itself need not be read.
 *   row_begin, row_end : 0 <= row_begin <= row_end < 2^31.
 *   K, stream, out : as in spmm_plan_create. Synchronous.
 * The plan's rows are local: M = row_end - row_begin, and C / argmax passed to
 * spmm_run are [M, N]. col and val passed to spmm_run, spmm_run_ex,
 * spmm_plan_validate_cols and spmm_transpose are the WHOLE matrix's arrays
 * (the plan reads its rows' entries from offset rowptr[row_begin]); B is the
 * whole K x N matrix. Column locality is measured against the global row, so
 * a banded matrix keeps its banded routing when the range starts on a
 * multiple of the WINDOW family's tile rows (256 covers every tile shape);
 * the BLOCK family needs row_begin == 0. Returns SPMM_ERR_INVALID_INPUT when
 * the copied entries decrease or rowptr[row_begin] < 0.
 */
spmm_status spmm_plan_create_range(const int32_t *rowptr, int64_t row_begin, int64_t row_end,
                                   int64_t K, void *stream, spmm_plan_t *out);

/*
 * spmm_partition_rows -- contiguous row ranges for `parts` workers, balanced
 * by work (pure host code; no CUDA call).
 *   rowptr     : HOST, int32 [M+1], a CSR row-pointer array (rowptr[0] == 0,
 *                non-decreasing; checked, SPMM_ERR_INVALID_INPUT otherwise).
 *   M          : rows, 0 <= M < 2^31.
 *   parts      : workers, >= 1.
 *   align_rows : every inner bound is a multiple of this (>= 1; 256 keeps
 *                banded ranges eligible for the WINDOW family).
 *   bounds     : HOST, int64 [parts + 1], receives 0 = b_0 <= b_1 <= ... <=
 *                b_parts = M; worker q owns rows [b_q, b_{q+1}).
 * A row's work is its entry count plus one (its output row). Bound q is the
 * first row whose prefix work reaches q/parts of the total, rounded to the
 * nearest multiple of align_rows and kept in order, so no row is split and a
 * heavy row stays whole on one worker. The objective is the block-workload
 * balance (maximum over average block work) of "Dual-Metric Partitioning with
 * Adaptive Kernel Execution for Efficient GCN Acceleration", section
 * "Adaptive Data Partitioning", with row degree as the width metric; its
 * random-walk density term and its reordering of nodes are not used, so each
 * worker's rows stay contiguous and C needs no permutation.
 */
spmm_status spmm_partition_rows(const int32_t *rowptr, int64_t M, int32_t parts,
                                int64_t align_rows, int64_t *bounds);

/*
 * spmm_run -- C = reduce_j A[i,j] * B[j,:] for every row i (asynchronous).
 *   col    : device, int32 [nnz], every value in [0, K). Not checked here (use
 *            spmm_plan_validate_cols once per graph); an out-of-range column
 *            is undefined behaviour.
 *   val    : device, fp32 [nnz], or NULL for an unweighted adjacency (every
 *            stored entry is 1 and the value load is skipped).
 *   B      : device, fp32 [K, N] row-major, contiguous.
 *   N      : feature width, N >= 0. N == 0 or M == 0 returns SPMM_OK with no launch.
 *   reduce : SPMM_SUM, SPMM_MEAN (divide by the row's stored-entry count,
 *            empty row -> 0) or SPMM_MAX (max over fp32 products, ties to the
 *            smallest column, empty row -> 0 and argmax -1).
 *   C      : device, fp32 [M, N] row-major, written once per element.
 *   argmax : device, int32 [M, N] (SPMM_MAX only; may be NULL to skip it).
 * 128-bit loads are used when N % 4 == 0 and B and C are 16-byte aligned;
 * otherwise the scalar path runs (same results). Grows the plan's workspace
 * with cudaMalloc when the heavy-row split or the open rows of the SEGMENT,
 * GATHER or STREAM families need more than it holds; the first GATHER or
 * STREAM product builds the plan's per-entry row ids (4 bytes per entry); use
 * spmm_plan_reserve beforehand to keep both out of timed or captured
 * regions. The first BLOCK product prepares the plan's diagonal blocks
 * (spmm_plan_prepare_blocks beforehand does the same).
 * (ParamSpMM section 2, Algorithm 1; graph-spmm model card, "Method".)
 */
spmm_status spmm_run(spmm_plan_t plan, const int32_t *col, const float *val, const float *B,
                     int64_t N, spmm_reduce reduce, float *C, int32_t *argmax, void *stream);

/*
 * spmm_run_ex -- spmm_run with a fused epilogue on every output element. A GCN
 * layer is the aggregation SpMM followed by the node update ("Dual-Metric
 * Partitioning with Adaptive Kernel Execution for Efficient GCN Acceleration",
 * introduction); here the bias and the activation are applied where C is
 * written, so C makes one trip to memory:
 *   C[i,k] = act(R[i,k] + bias[k])
 * with R the reduction's value as spmm_run defines it (empty rows included:
 * R = 0), the addition in fp32 (round to nearest) and act applied after it.
 *   bias : device, fp32 [N], or NULL for no bias.
 *   act  : SPMM_ACT_NONE, or SPMM_ACT_RELU (x > 0 ? x : +0).
 * argmax (SPMM_MAX) is the reduction's and is not affected. Everything else,
 * including the error behaviour, is as in spmm_run; an unknown act returns
 * SPMM_ERR_INVALID_ARG. spmm_run(...) is spmm_run_ex(..., NULL, SPMM_ACT_NONE, ...).
 */
spmm_status spmm_run_ex(spmm_plan_t plan, const int32_t *col, const float *val, const float *B,
                        int64_t N, spmm_reduce reduce, const float *bias, spmm_activation act,
                        float *C, int32_t *argmax, void *stream);

/*
 * spmm_plan_reserve -- allocate the workspace spmm_run needs for (N, reduce)
 * now, and when that product goes to the GATHER or STREAM family, build the
 * plan's per-entry row ids. Synchronous (cudaMalloc). Returns SPMM_ERR_OOM on
 * failure.
 */
spmm_status spmm_plan_reserve(spmm_plan_t plan, int64_t N, spmm_reduce reduce);

/*
 * spmm_plan_validate_cols -- check that every col[p], p < nnz, lies in [0, K),
 * and measure the column spread |col[p] - row(p)| (a log2 histogram) from
 * which the router decides whether the WINDOW family applies. Until this has
 * been called for a plan, the WINDOW family is not used.
 *   col : device, int32 [nnz]. Synchronous on `stream`.
 * Returns SPMM_ERR_INVALID_INPUT if any entry is out of range.
 */
spmm_status spmm_plan_validate_cols(spmm_plan_t plan, const int32_t *col, void *stream);

/*
 * spmm_plan_prepare_blocks -- the BLOCK family's per-plan preparation (RA-SpMM,
 * "tensor-core SpMM with per-matrix preprocessing": A is fixed, so its dense
 * blocks are built once and reused by every product). For every 128-row tile
 * the 256-column diagonal block is densified (duplicates added in CSR order,
 * fp32) and split into TF32 hi and lo operand pieces in the tensor cores'
 * layout; the entries outside the diagonal blocks are copied, in CSR order,
 * into a compact CSR. Plan-owned device memory: 256 KB per 128-row tile plus
 * 4 (M + 1) + 8 (4 unweighted) bytes per outside entry (spmm_plan_info's
 * block_bytes).
 *   col, val : device, the plan's graph (as for spmm_run; val NULL when A is
 *              unweighted). The pieces are a copy: after changing col or val,
 *              prepare again.
 * spmm_run prepares on first use of the BLOCK family (and again when the
 * flavour of A, weighted or not, changes), so this call only moves that cost
 * out of the first product. Synchronous. SPMM_ERR_UNSUPPORTED for a
 * row-range plan; SPMM_ERR_OOM when the device is full.
 */
spmm_status spmm_plan_prepare_blocks(spmm_plan_t plan, const int32_t *col, const float *val,
                                     void *stream);

/*
 * spmm_plan_sync -- wait for `stream`, then report any error a kernel of this
 * plan recorded on the device (SPMM_ERR_TIMEOUT when a bounded wait gave up)
 * and clear it. Synchronous.
 */
spmm_status spmm_plan_sync(spmm_plan_t plan, void *stream);

/*
 * spmm_plan_describe -- descriptors plus the routing decision spmm_run will
 * take for (N, reduce) with 16-byte aligned B, C, col and val and a val array
 * present. Host only, no CUDA call.
 */
spmm_status spmm_plan_describe(spmm_plan_t plan, int64_t N, spmm_reduce reduce,
                               spmm_plan_info *out);

/*
 * spmm_plan_set_family -- pin the light-row family (SPMM_FAMILY_AUTO restores
 * the router) and the heavy-row threshold (t_split <= 0 restores the default;
 * a threshold above INT32_MAX is taken as INT32_MAX, i.e. no row is split;
 * a new threshold rebuilds the heavy-row tables, synchronously on the legacy
 * default stream). `family` is an spmm_family value, SPMM_FAMILY_AUTO to
 * SPMM_FAMILY_STREAM, else SPMM_ERR_INVALID_ARG. When a pinned family's
 * conditions (see spmm_family) do not hold for a product, that product runs
 * as WARPROW (pinned COLTILE, SEGMENT, GATHER, STREAM) or as the router
 * would choose (pinned WINDOW, BLOCK). For tests and benchmarks of
 * individual families.
 */
spmm_status spmm_plan_set_family(spmm_plan_t plan, int family, int64_t t_split);

/*
 * spmm_route -- the router as a pure host function. Reads the descriptor
 * fields of *desc (M, K, nnz, d_max, dbar, cv, t_split, chunk, n_heavy,
 * n_chunks, band_w, band_cover, blk_intra, row0, seg_tiles) and, with
 * family_override as spmm_plan_set_family's `family`, fills the launch-shape fields of *out for
 * (N, reduce) on a GPU with `num_sms` SMs. `aligned` is a bit mask: bit 0 set
 * when B, C (and argmax) are 16-byte aligned, bit 1 set when col (and val)
 * are 16-byte aligned, bit 2 set when there is no val array (unweighted).
 * No CUDA call. (RA-SpMM "routing rules": first matching rule wins.)
 */
spmm_status spmm_route(const spmm_plan_info *desc, int64_t N, spmm_reduce reduce, int aligned,
                       int num_sms, int family_override, spmm_plan_info *out);

/*
 * spmm_default_t_split -- the heavy-row threshold the plan uses for a graph of
 * `nnz` entries on `num_sms` SMs: nnz / (128 num_sms) clamped to [256, 512]
 * (pure host function).
 */
int64_t spmm_default_t_split(int64_t M, int64_t nnz, int num_sms);

/*
 * spmm_run_noalloc -- the product of spmm_run, for callers that cannot
 * allocate device memory: no plan, and no cudaMalloc / cudaFree or other
 * allocating call on any path. The pages have no counterpart of this call;
 * it exists for callers whose device memory is owned by another allocator
 * (a framework's caching pool that a stray cudaMalloc would fragment or
 * exhaust) and for serving loops that must not allocate after start-up
 * (cudaMalloc and cudaFree synchronise the device and can fail at any time).
 *   rowptr, col, val, B, C, argmax : as in spmm_plan_create and spmm_run,
 *            all device pointers owned by the caller.
 *   M, K, N, reduce, stream        : as in spmm_plan_create and spmm_run.
 * Rows are reduced by the WARPROW family; rows longer than
 * spmm_default_t_split(M, nnz, SMs) are split into chunks whose partials go to
 * a file-scope device array of 64 MiB that every GPU which loads the library
 * holds until the process exits. At most 65,536 split rows, 262,144 chunks and
 * chunks x N x 4 bytes of partials (x 2 for SPMM_MAX) up to about 60 MiB fit
 * in it; larger inputs return SPMM_ERR_UNSUPPORTED before any product kernel
 * runs. rowptr[0] != 0 or a decreasing rowptr returns SPMM_ERR_INVALID_INPUT.
 * Partly synchronous: nnz and the split-row counts are read back to the host
 * (draining `stream`) before the product is enqueued. The split rows are found
 * by three small launches over blocks of at least 4,096 rows.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress; make that first call before any stream capture.
 * Every call shares the one array and it keeps the last call's contents:
 * calls whose GPU work overlaps (other streams, other host threads) race and
 * must be serialised by the caller.
 */
spmm_status spmm_run_noalloc(const int32_t *rowptr, const int32_t *col, const float *val,
                             const float *B, int64_t M, int64_t K, int64_t N, spmm_reduce reduce,
                             float *C, int32_t *argmax, void *stream);

/*
 * spmm_transpose -- A^T in CSR, for the backward of a product (graph-spmm
 * model card, "Requirements and limits": the gradient of a sum aggregation
 * with respect to B is the product with the transposed adjacency, A^T . dC).
 *   plan    : the plan of A (M x K).
 *   col     : device, int32 [nnz], every value in [0, K) (validated columns;
 *             an out-of-range column gives an undefined result but no fault).
 *   val     : device, fp32 [nnz], or NULL for an unweighted A.
 *   scale_mean : nonzero -> the value of entry (i, j) becomes a_ij / d_i
 *             (1 / d_i when val is NULL), computed in fp64 and rounded once to
 *             fp32, d_i the stored-entry count of row i: then a product with
 *             the result is the backward of the mean.
 *   rowptrT : device, int32 [K + 1], written.
 *   colT    : device, int32 [nnz], written: row j of A^T lists the rows i of
 *             the entries (i, j) of A in increasing i, and the entries of one
 *             row i in their CSR order (a stable sort of the entries by column).
 *   valT    : device, fp32 [nnz], written (the entries' values in colT's
 *             order), or NULL to skip the values. Required when val != NULL or
 *             scale_mean; when val is NULL and valT is not, every value is 1
 *             (or 1 / d_i).
 * Each output element is a pure function of the input: the sort places every
 * entry by exact integer ranks, with no atomics. Synchronous: temporaries of
 * about 5 x 4 x nnz bytes are allocated with cudaMalloc and freed before the
 * call returns. SPMM_ERR_OOM if they do not fit.
 */
spmm_status spmm_transpose(spmm_plan_t plan, const int32_t *col, const float *val, int scale_mean,
                           int32_t *rowptrT, int32_t *colT, float *valT, void *stream);

/*
 * spmm_maxpool_backward -- the gradient of spmm_max with respect to B
 * (graph-spmm model card, "API": spmm_max returns the argmax so that the
 * max-pool backward can route the gradient to the winning column;
 * "Correctness": duplicated pairs are legal CSR).
 *   planT  : the plan of A^T (K x M), built from spmm_transpose's rowptrT.
 *   colT, valT : spmm_transpose's output (valT unscaled, or NULL when A is
 *            unweighted).
 *   B      : device, fp32 [K, N], the forward's B. Required when valT is not
 *            NULL (it decides which copy of a duplicated pair won); may be
 *            NULL for an unweighted A.
 *   argmax : device, int32 [M, N], as written by spmm_run with SPMM_MAX.
 *   dC     : device, fp32 [M, N], the gradient of C.
 *   dB     : device, fp32 [K, N], written once per element:
 *            dB[j, c] = sum over the rows i with argmax[i, c] == j of
 *            a_w * dC[i, c], where w is the stored entry of row i whose
 *            product won the forward maximum: among the copies of (i, j), the
 *            one with the largest fp32 product a * B[j, c], the first in CSR
 *            order on equal products (so an unweighted duplicated pair passes
 *            dC once). Accumulated in fp32 in increasing i; 0 where no row
 *            chose j. Rows of A^T longer than planT's split threshold (hub
 *            columns of A) are cut into planT's chunks: each chunk is summed
 *            in increasing i, then the chunks in order (no atomics;
 *            reproducible).
 * Asynchronous, except that the first call with split rows at a given N
 * grows planT's workspace with cudaMalloc (spmm_plan_reserve(planT, N,
 * SPMM_SUM) beforehand keeps allocation out). 128-bit loads when N % 4 == 0
 * and B, argmax, dC and dB are 16-byte aligned. SPMM_ERR_INVALID_ARG when a
 * required pointer is NULL.
 */
spmm_status spmm_maxpool_backward(spmm_plan_t planT, const int32_t *colT, const float *valT,
                                  const float *B, const int32_t *argmax, const float *dC,
                                  int64_t N, float *dB, void *stream);

/*
 * spmm_check_wait_timeout -- diagnostic of the failure path. Every spin-wait in
 * the library's kernels is bounded: when it gives up it records a timeout in
 * the plan's error words and the kernel returns (no trap), and
 * spmm_plan_sync then reports SPMM_ERR_TIMEOUT. This call runs, on `stream`,
 * one kernel whose wait nothing completes, with a limit of `limit_us`
 * microseconds (1 .. 10^7), then returns what spmm_plan_sync returns:
 * SPMM_ERR_TIMEOUT when the path works. The plan and the CUDA context stay
 * usable afterwards. Synchronous.
 */
spmm_status spmm_check_wait_timeout(spmm_plan_t plan, int64_t limit_us, void *stream);

/* spmm_plan_destroy -- free the plan and everything it owns. NULL is a no-op. */
spmm_status spmm_plan_destroy(spmm_plan_t plan);

/* spmm_status_string -- static description of a status code. */
const char *spmm_status_string(spmm_status status);

/* spmm_launch_count -- kernels this library has launched in this process. */
uint64_t spmm_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SPMM_H */
