// COLTILE family: wide N. A CTA of 8 warps owns RB consecutive rows and, for
// each of them, WPR warps that each own a 128-column tile (32 lanes x float4).
// The entries of the CTA's light rows are staged into shared memory chunk by
// chunk, once per CTA: the 16-byte aligned middle of a row segment of at least
// kBulkMin entries arrives by a 1-D bulk copy, the rest by cooperative loads.
// Each warp then reads its row's (col, val) pairs by shared-memory broadcast and
// gathers 512-byte slices of the B rows, four in flight per lane. So the WPR
// column-tile warps of a row share one read of its col/val (GE-SpMM section
// III-B, coalesced row caching, and III-C, warp merging, here as a CTA-wide
// stage), and the tiles of one row are covered by one CTA.
// In the compacted stage every row starts at an index congruent to its first
// global entry modulo 4, so a shared-memory offset and a global offset share
// their 16-byte alignment and the middle of a segment can be bulk-copied.
// Rows longer than t_split are left to the heavy-row split.
#include "common.cuh"
#include "tma.cuh"

namespace spmm {

namespace {

constexpr int kCtThreads = 256;
constexpr int kCtWarps = kCtThreads / kWarp;
constexpr int kCtChunk = 2048;     // staged entries per chunk (multiple of 4)
constexpr int kBulkMin = 64;       // shortest aligned middle worth a bulk copy

template <int RED, bool HAS_VAL>
__global__ void __launch_bounds__(kCtThreads) k_coltile(const RunArgs a, int wpr, int bulk_ok) {
    __shared__ __align__(16) int s_col[kCtChunk];
    __shared__ __align__(16) float s_val[HAS_VAL ? kCtChunk : 4];
    __shared__ int s_p0[kCtWarps], s_start[kCtWarps], s_end[kCtWarps], s_d[kCtWarps];
    __shared__ int s_total;
    __shared__ __align__(8) uint64_t s_bar;

    const int rb = kCtWarps / wpr;                  // rows per CTA
    const int64_t r0 = (int64_t)blockIdx.x * rb;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x & (kWarp - 1);

    if (warp == 0) {
        // compacted layout of the block's light rows (padding keeps residues mod 4):
        // lane q < rb loads row q's bounds, lane 0 lays the rows out
        int p0 = 0, d = 0;
        const int64_t row = r0 + lane;
        if (lane < rb && row < a.M) {
            p0 = a.rowptr[row];
            d = a.rowptr[row + 1] - p0;
        }
        const int len = (lane < rb && row < a.M && d <= a.t_split) ? d : 0;
        int pos = 0, my_start = 0;
        for (int q = 0; q < kCtWarps; ++q) {
            const int pq = __shfl_sync(0xffffffffu, p0, q);
            const int lq = __shfl_sync(0xffffffffu, len, q);
            if (q < rb) {
                pos += (pq - pos) & 3;
                if (lane == q) my_start = pos;
                pos += lq;
            }
        }
        if (lane < rb) {
            s_p0[lane] = p0;
            s_d[lane] = d;
            s_start[lane] = my_start;
            s_end[lane] = my_start + len;
        }
        if (lane == 0) {
            s_total = pos;
            mbar_init(&s_bar, 1);
            mbar_init_fence();
        }
    }
    __syncthreads();

    const int rs = warp / wpr;                      // this warp's row slot
    const int tile = blockIdx.y * wpr + warp % wpr; // this warp's 128-column tile
    const int c = tile * 128 + 4 * lane;
    const bool row_ok = rs < rb && r0 + rs < a.M && s_d[rs] <= a.t_split;
    const bool active = row_ok && c < a.N;
    const float *Bv = a.B + min(c, a.N - 4);
    const int64_t N = a.N;
    Acc<4, RED, HAS_VAL> acc;
    acc.init();

    const int total = s_total;
    for (int c0 = 0, chunk = 0; c0 < total; c0 += kCtChunk, ++chunk) {
        const int c1 = min(total, c0 + kCtChunk);
        // bulk copies of aligned segment middles (thread 0 plans and issues)
        if (threadIdx.x == 0) {
            uint32_t tx = 0;
            if (bulk_ok) {
                for (int q = 0; q < rb; ++q) {
                    const int b = max(s_start[q], c0), e = min(s_end[q], c1);
                    const int bm = (b + 3) & ~3, em = e & ~3;
                    if (em - bm >= kBulkMin) tx += (uint32_t)(em - bm) * 4u * (HAS_VAL ? 2u : 1u);
                }
            }
            // order earlier generic reads of the stage before the async writes
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&s_bar, tx);
            if (tx) {
                for (int q = 0; q < rb; ++q) {
                    const int b = max(s_start[q], c0), e = min(s_end[q], c1);
                    const int bm = (b + 3) & ~3, em = e & ~3;
                    if (em - bm < kBulkMin) continue;
                    const int g = s_p0[q] + (bm - s_start[q]);     // global entry of bm
                    bulk_g2s(&s_col[bm - c0], a.col + g, (uint32_t)(em - bm) * 4u, &s_bar);
                    if (HAS_VAL)
                        bulk_g2s(&s_val[bm - c0], a.val + g, (uint32_t)(em - bm) * 4u, &s_bar);
                }
            }
        }
        // everything else: cooperative loads
        for (int q = c0 + threadIdx.x; q < c1; q += kCtThreads) {
            int r = -1;
            for (int t = 0; t < rb; ++t)
                if (q >= s_start[t] && q < s_end[t]) r = t;
            if (r < 0) continue;                    // padding between rows
            if (bulk_ok) {
                const int b = max(s_start[r], c0), e = min(s_end[r], c1);
                const int bm = (b + 3) & ~3, em = e & ~3;
                if (em - bm >= kBulkMin && q >= bm && q < em) continue;   // bulk-copied
            }
            const int g = s_p0[r] + (q - s_start[r]);
            s_col[q - c0] = ld_stream(a.col + g);
            if (HAS_VAL) s_val[q - c0] = ld_stream(a.val + g);
        }
        const bool ok = mbar_wait(&s_bar, (uint32_t)chunk & 1u, a.err);
        if (!__syncthreads_and(ok)) {
            // a copy did not land in time (error recorded): wait once more, bounded,
            // so that no copy is still writing into this CTA's shared memory
            if (threadIdx.x == 0) mbar_wait(&s_bar, (uint32_t)chunk & 1u, a.err);
            __syncthreads();
            return;
        }

        if (row_ok) {
            const int b = max(s_start[rs], c0) - c0, e = min(s_end[rs], c1) - c0;
            int q = b;
            for (; q + 4 <= e; q += 4) {
                int j[4];
                float w[4], x[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    j[u] = s_col[q + u];
                    w[u] = HAS_VAL ? s_val[q + u] : 1.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) ld_vec<4>(Bv + (int64_t)j[u] * N, x[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc.add(w[u], j[u], x[u]);
            }
            for (; q < e; ++q) {
                const int j = s_col[q];
                float x[4];
                ld_vec<4>(Bv + (int64_t)j * N, x);
                acc.add(HAS_VAL ? s_val[q] : 1.0f, j, x);
            }
        }
        __syncthreads();                            // the stage is rewritten next chunk
    }
    if (!active) return;
    float out[4];
    int arg[4];
    acc.finish(s_d[rs], out, arg);
    epilogue<4>(a, c, out);
    const int64_t i = r0 + rs;
    st_vec<4>(a.C + i * N + c, out);
    if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + i * N + c, arg);
}

template <int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, int wpr, int tiles_y, int bulk_ok, cudaStream_t s) {
    const int rb = kCtWarps / wpr;
    const int64_t blocks = (a.M + rb - 1) / rb;
    k_coltile<RED, HAS_VAL><<<dim3((unsigned)blocks, (unsigned)tiles_y), kCtThreads, 0, s>>>(
        a, wpr, bulk_ok);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

// wpr: warps per row (1, 2, 4 or 8); tiles_y: grid.y (groups of wpr tiles).
cudaError_t launch_coltile(const RunArgs &a, int wpr, int tiles_y, int reduce, bool has_val,
                           bool bulk_ok, cudaStream_t s) {
    const int b = bulk_ok ? 1 : 0;
#define SPMM_RED(R)                                                       \
    return has_val ? go<R, true>(a, wpr, tiles_y, b, s) : go<R, false>(a, wpr, tiles_y, b, s);
    switch (reduce) {
        case SPMM_SUM: SPMM_RED(SPMM_SUM)
        case SPMM_MEAN: SPMM_RED(SPMM_MEAN)
        case SPMM_MAX: SPMM_RED(SPMM_MAX)
    }
#undef SPMM_RED
    return cudaErrorInvalidValue;
}

}  // namespace spmm
