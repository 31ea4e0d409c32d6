// WINDOW family: persistent, warp-specialised SpMM for graphs with column
// locality (RA-SpMM's community/locality regime), where most entries of row i
// lie within |j - i| <= W.
//
// Each CTA owns a contiguous range of row tiles (R rows each) and one column
// tile of cw columns. A producer warp streams, per tile and through a
// three-stage mbarrier pipeline:
//   * the tile's row pointers (plain loads),
//   * its col / val segment (1-D bulk copies, 16-byte aligned part),
//   * the B rows [r1 + W_prev, r1 + W) that enter the tile's window
//     [r0 - W, r1 + W) -- bulk copies into a ring buffer of `cap` B rows in
//     shared memory (cap >= 3R + 2W, so the rows of the two tiles still in
//     flight are never overwritten).
// Sixteen consumer warps (L lanes per row, one row per lane group) read the
// entries from shared memory and the gathered B rows from the ring; an entry
// whose column falls outside the window is read from global memory instead.
// Every B row is thus fetched from L2/HBM once per CTA range (plus a 2W halo)
// instead of once per entry, and no consumer waits on a global gather.
// Rows longer than t_split are left to the heavy-row split, as everywhere.
// Results match the other families' order: entries in CSR order per lane,
// fp32 FMA, written once.
#include "common.cuh"
#include "tma.cuh"

namespace spmm {

constexpr int kWinStages = 3;
constexpr int kWinConsumerWarps = 16;
constexpr int kWinThreads = (kWinConsumerWarps + 1) * kWarp;

template <int L, int RED, bool HAS_VAL>
__global__ void __launch_bounds__(kWinThreads, 1) k_window(const RunArgs a, const WinShape w) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kWinStages;
    int *meta = reinterpret_cast<int *>(smem + w.off_meta);      // [S][4]
    int *rp = reinterpret_cast<int *>(smem + w.off_rp);          // [S][Rp]
    int *scol = reinterpret_cast<int *>(smem + w.off_col);       // [S][ecap]
    float *sval = reinterpret_cast<float *>(smem + w.off_val);   // [S][ecap]
    float *ring = reinterpret_cast<float *>(smem + w.off_ring);  // [cap][cw]

    const int col0 = blockIdx.y * w.cw;
    const int cw_eff = min(w.cw, a.N - col0);
    const int64_t N = a.N;
    const int64_t tiles = (a.M + w.R - 1) / w.R;
    const int64_t t_begin = tiles * blockIdx.x / gridDim.x;
    const int64_t t_end = tiles * (blockIdx.x + 1) / gridDim.x;
    const int n_tiles = (int)(t_end - t_begin);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWinStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWinConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();

    const int warp = threadIdx.x / kWarp;
    const int lane = threadIdx.x & (kWarp - 1);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int64_t loaded_hi = 0;   // ring holds B rows [loaded_hi - cap, loaded_hi)
        int issued = 0;
        for (int k = 0; k < n_tiles; ++k) {
            const int s = k % kWinStages;
            const uint32_t use = (uint32_t)(k / kWinStages);
            if (use > 0) {
                const bool ok = mbar_wait(&empty[s], (use - 1) & 1, a.err);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            const int64_t r0 = (t_begin + k) * w.R;
            const int64_t r1 = min(r0 + w.R, a.M);
            const int nr = (int)(r1 - r0);
            int *rps = rp + s * w.Rp;
            for (int q = lane; q <= nr; q += kWarp) rps[q] = ld_stream(a.rowptr + r0 + q);
            __syncwarp();
            const int seg_b = rps[0], seg_e = rps[nr];
            const int s_al = seg_b & ~3;
            const bool overflow = (seg_e - s_al) > w.ecap;
            int e_cp = s_al;                 // entries [s_al, e_cp) arrive by bulk copy
            if (!overflow) {
                e_cp = max(s_al, min((seg_e + 3) & ~3, a.nnz4));
                // the last < 4 entries of the whole array: plain loads
                for (int p = e_cp + lane; p < seg_e; p += kWarp) {
                    scol[s * w.ecap + (p - s_al)] = ld_stream(a.col + p);
                    if (HAS_VAL) sval[s * w.ecap + (p - s_al)] = ld_stream(a.val + p);
                }
            }
            const int64_t win_lo = max(r0 - (int64_t)w.W, (int64_t)0);
            const int64_t win_hi = min(r1 + (int64_t)w.W, a.K);
            const int64_t lo = (k == 0) ? win_lo : max(loaded_hi, win_lo);
            const int64_t hi = max(win_hi, lo);
            if (lane == 0) {
                meta[4 * s + 0] = s_al;
                meta[4 * s + 1] = overflow ? 1 : 0;
                meta[4 * s + 2] = (int)win_lo;
                meta[4 * s + 3] = (int)win_hi;
            }
            const uint32_t seg_bytes = (uint32_t)(e_cp - s_al) * 4u;
            const uint32_t tx = seg_bytes * (HAS_VAL ? 2u : 1u) +
                                (uint32_t)(hi - lo) * (uint32_t)cw_eff * 4u;
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], tx);
            __syncwarp();
            if (seg_bytes) {
                if (lane == 0) bulk_g2s(scol + s * w.ecap, a.col + s_al, seg_bytes, &full[s]);
                if (HAS_VAL && lane == 1) bulk_g2s(sval + s * w.ecap, a.val + s_al, seg_bytes, &full[s]);
            }
            if (w.cw == a.N) {
                // ring rows are whole B rows: one copy per run up to the ring's wrap
                if (lane == 2) {
                    int64_t j = lo;
                    while (j < hi) {
                        const int slot = (int)(j % w.cap);
                        const int64_t run = min(hi - j, (int64_t)(w.cap - slot));
                        bulk_g2s(ring + (int64_t)slot * w.cw, a.B + j * N,
                                 (uint32_t)(run * N * 4), &full[s]);
                        j += run;
                    }
                }
            } else {
                for (int64_t j = lo + lane; j < hi; j += kWarp)
                    bulk_g2s(ring + (j % w.cap) * w.cw, a.B + j * N + col0,
                             (uint32_t)cw_eff * 4u, &full[s]);
            }
            loaded_hi = max(loaded_hi, hi);
            issued = k + 1;
        }
        // never leave while copies this warp issued may still be landing
        for (int k = max(0, issued - kWinStages); k < issued; ++k)
            mbar_wait(&full[k % kWinStages], (uint32_t)(k / kWinStages) & 1, a.err);
        return;
    }

    // -------------------------------------------------------------- consumers
    constexpr int kGroups = kWinConsumerWarps * kWarp / L;
    const int ct = threadIdx.x - kWarp;
    const int grp = ct / L;
    const int li = ct % L;
    const int c = col0 + 4 * li;               // first of this lane's 4 columns
    const bool active = c < a.N;
    const float *Bg = a.B + min(c, a.N - 4);   // global fallback (clamped for idle lanes)
    for (int k = 0; k < n_tiles; ++k) {
        const int s = k % kWinStages;
        const bool ok = mbar_wait(&full[s], (uint32_t)(k / kWinStages) & 1, a.err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int64_t r0 = (t_begin + k) * w.R;
        const int nr = (int)(min(r0 + w.R, a.M) - r0);
        const int s_al = meta[4 * s + 0];
        const bool overflow = meta[4 * s + 1] != 0;
        const int win_lo = meta[4 * s + 2];
        const int win_hi = meta[4 * s + 3];
        const int m0 = win_lo % w.cap;
        const int *rps = rp + s * w.Rp;
        const int *cs = scol + s * w.ecap - s_al;
        const float *vs = sval + s * w.ecap - s_al;
        for (int rr = grp; rr < nr; rr += kGroups) {
            const int p0 = rps[rr], p1 = rps[rr + 1];
            const int d = p1 - p0;
            if (d > a.t_split) continue;
            Acc<4, RED, HAS_VAL> acc;
            acc.init();
            for (int p = p0; p < p1; p += 4) {
                int j[4];
                float wv[4], b[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int q = min(p + u, p1 - 1);
                    j[u] = overflow ? ld_stream(a.col + q) : cs[q];
                    wv[u] = HAS_VAL ? (overflow ? ld_stream(a.val + q) : vs[q]) : 1.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (j[u] >= win_lo && j[u] < win_hi) {
                        int slot = j[u] - win_lo + m0;
                        if (slot >= w.cap) slot -= w.cap;
                        const float4 v =
                            *reinterpret_cast<const float4 *>(ring + (int64_t)slot * w.cw + 4 * li);
                        b[u][0] = v.x; b[u][1] = v.y; b[u][2] = v.z; b[u][3] = v.w;
                    } else {
                        ld_vec<4>(Bg + (int64_t)j[u] * N, b[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (p + u < p1) acc.add(wv[u], j[u], b[u]);
            }
            if (active) {
                float out[4];
                int arg[4];
                acc.finish(d, out, arg);
                const int64_t i = r0 + rr;
                st_vec<4>(a.C + i * N + c, out);
                if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + i * N + c, arg);
            }
        }
        __syncwarp();
        if ((threadIdx.x & (kWarp - 1)) == 0) mbar_arrive(&empty[s]);
    }
}

// ---------------------------------------------------------------- host side
bool window_shape(int64_t M, int64_t K, int64_t N, double dbar, int64_t W, bool has_val,
                  int lanes, WinShape *o) {
    if (lanes < 2 || lanes > 32 || W < 0) return false;
    WinShape w{};
    w.R = kWinConsumerWarps * kWarp / lanes;
    w.W = (int)W;
    w.cw = 4 * lanes;
    w.cap = kWinStages * w.R + 2 * (int)W;
    w.Rp = (w.R + 1 + 3) & ~3;
    int64_t ecap = (int64_t)(w.R * dbar * 1.25) + 64;
    ecap = std::min<int64_t>(4096, std::max<int64_t>(256, (ecap + 3) & ~3));
    w.ecap = (int)ecap;
    int off = 2 * kWinStages * 8;
    w.off_meta = off;
    off += kWinStages * 16;
    off = (off + 15) & ~15;
    w.off_rp = off;
    off += kWinStages * w.Rp * 4;
    off = (off + 15) & ~15;
    w.off_col = off;
    off += kWinStages * w.ecap * 4;
    w.off_val = off;
    if (has_val) off += kWinStages * w.ecap * 4;
    off = (off + 127) & ~127;
    w.off_ring = off;
    off += w.cap * w.cw * 4;
    w.smem_bytes = off;
    (void)M; (void)K; (void)N;
    *o = w;
    return true;
}

namespace {
template <int L, int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, const WinShape &w, int grid_x, int tiles, cudaStream_t s) {
    auto kern = k_window<L, RED, HAS_VAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         w.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)grid_x, (unsigned)tiles), kWinThreads, w.smem_bytes, s>>>(a, w);
    count_launch();
    return cudaGetLastError();
}

template <int RED, bool HAS_VAL>
cudaError_t by_lanes(const RunArgs &a, const WinShape &w, int lanes, int gx, int tiles,
                     cudaStream_t s) {
    switch (lanes) {
        case 2: return go<2, RED, HAS_VAL>(a, w, gx, tiles, s);
        case 4: return go<4, RED, HAS_VAL>(a, w, gx, tiles, s);
        case 8: return go<8, RED, HAS_VAL>(a, w, gx, tiles, s);
        case 16: return go<16, RED, HAS_VAL>(a, w, gx, tiles, s);
        case 32: return go<32, RED, HAS_VAL>(a, w, gx, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_window(const RunArgs &a, const WinShape &w, int lanes, int reduce, bool has_val,
                          int grid_x, int tiles, cudaStream_t s) {
#define SPMM_RED(R)                                                            \
    return has_val ? by_lanes<R, true>(a, w, lanes, grid_x, tiles, s)          \
                   : by_lanes<R, false>(a, w, lanes, grid_x, tiles, s);
    switch (reduce) {
        case SPMM_SUM: SPMM_RED(SPMM_SUM)
        case SPMM_MEAN: SPMM_RED(SPMM_MEAN)
        case SPMM_MAX: SPMM_RED(SPMM_MAX)
    }
#undef SPMM_RED
    return cudaErrorInvalidValue;
}

}  // namespace spmm
