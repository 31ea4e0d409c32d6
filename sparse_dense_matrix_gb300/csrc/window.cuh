// WINDOW family: persistent, warp-specialised SpMM for graphs with column
// locality (RA-SpMM's community/locality regime), where most entries of row i
// lie within |j - i| <= W.
//
// Each CTA owns a contiguous range of row tiles (R rows each) and one column
// tile of cw columns. A producer warp streams, per tile and through an
// S-stage mbarrier pipeline (3 <= S <= 8, as deep as shared memory allows):
//   * the tile's row pointers (a bulk copy from the plan's padded copy; the
//     tiles' segment bounds are loaded in batches of 32 tiles, one batch ahead),
//   * its col / val segment (1-D bulk copies of the 16-byte aligned part),
//   * the B rows entering the tile's window [r0 - W, r1 + W): into a ring of
//     `cap` B rows in shared memory (cap >= S R + 2W for S pipeline stages, so
//     rows of the tiles still in flight are never overwritten). Whole rows (cw == N) come by 1-D bulk
//     copies; a column slice (cw < N) comes by 2-D tensor copies of R x cw
//     boxes, with W and cap multiples of R so that boxes never wrap.
// Sixteen consumer warps (L lanes per row, two rows per lane group) read the
// entries from shared memory and the gathered B rows from the ring; an entry
// outside the window (possible only when not every entry is within W) is read
// from global memory instead. Every B row is thus fetched from L2/HBM once per
// CTA range (plus a 2W halo) rather than once per entry.
// Rows longer than t_split are left to the heavy-row split, as everywhere.
// Per lane the entries are accumulated in CSR order with fp32 FMA.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace spmm {

constexpr int kWinMaxStages = 8;
constexpr int kWinConsumerWarps = 16;
constexpr int kWinThreads = (kWinConsumerWarps + 1) * kWarp;

template <int L, int RED, bool HAS_VAL, bool CHECK, bool POW2>
__global__ void __launch_bounds__(kWinThreads, 1)
    k_window(const RunArgs a, const WinShape w, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 128-byte aligned base (tensor copies want 128-byte aligned destinations)
    unsigned char *smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kWinMaxStages;
    const int S = w.S;
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
        for (int s = 0; s < S; ++s) {
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
        int64_t loaded_hi = 0;   // B rows below loaded_hi have been requested
        int issued = 0;
        // Segment bounds: lane l holds rowptr[start of tile kb + l] for the current
        // batch of 32 tiles (bcur) and the next batch (bnxt); a batch is loaded 32
        // tiles before it is used, so no tile waits on a row-pointer load.
        auto tile_start = [&](int kk) {
            const int64_t q = min((t_begin + kk) * (int64_t)w.R, a.M);
            return ld_stream(a.rowptr + q);
        };
        int bcur = tile_start(min(lane, n_tiles));
        int bnxt = tile_start(min(kWarp + lane, n_tiles));
        for (int k = 0; k < n_tiles; ++k) {
            const int s = k % S;
            const uint32_t use = (uint32_t)(k / S);
            if (use > 0) {
                const bool ok = mbar_wait(&empty[s], (use - 1) & 1, a.err);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            const int64_t r0 = (t_begin + k) * w.R;
            const int64_t r1 = min(r0 + w.R, a.M);
            const int kl = k & (kWarp - 1);
            if (kl == 0 && k > 0) {
                bcur = bnxt;
                bnxt = tile_start(min(k + kWarp + lane, n_tiles));
            }
            const int seg_b = __shfl_sync(0xffffffffu, bcur, kl);
            const int seg_e = kl == kWarp - 1 ? __shfl_sync(0xffffffffu, bnxt, 0)
                                               : __shfl_sync(0xffffffffu, bcur, kl + 1);
            int *rps = rp + s * w.Rp;
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
            // window of this tile, and the B rows it adds to the ring
            const int64_t win_lo = max(r0 - (int64_t)w.W, (int64_t)0);
            const int64_t win_hi = min(r1 + (int64_t)w.W, a.K);
            int64_t lo = (k == 0) ? win_lo : max(loaded_hi, win_lo);
            int64_t hi = max(win_hi, lo);
            uint32_t ring_bytes;
            if (w.tmap) {                    // whole R-row boxes (multiples of R)
                hi = min((hi + w.R - 1) / w.R * w.R, (a.K + w.R - 1) / w.R * w.R);
                hi = max(hi, lo);
                ring_bytes = (uint32_t)((hi - lo) / w.R) * (uint32_t)w.R * (uint32_t)w.cw * 4u;
            } else {
                ring_bytes = (uint32_t)(hi - lo) * (uint32_t)cw_eff * 4u;
            }
            if (lane == 0) {
                meta[4 * s + 0] = s_al;
                meta[4 * s + 1] = overflow ? 1 : 0;
                meta[4 * s + 2] = (int)win_lo;
                meta[4 * s + 3] = (int)win_hi;
            }
            const uint32_t seg_bytes = (uint32_t)(e_cp - s_al) * 4u;
            const uint32_t rp_bytes = (uint32_t)w.Rp * 4u;
            const uint32_t tx = rp_bytes + seg_bytes * (HAS_VAL ? 2u : 1u) + ring_bytes;
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], tx);
            __syncwarp();
            // row pointers of the tile: the plan's copy is padded past rowptr[M]
            if (lane == 3) bulk_g2s(rps, a.rowptr + r0, rp_bytes, &full[s]);
            if (seg_bytes) {
                if (lane == 0) bulk_g2s(scol + s * w.ecap, a.col + s_al, seg_bytes, &full[s]);
                if (HAS_VAL && lane == 1) bulk_g2s(sval + s * w.ecap, a.val + s_al, seg_bytes, &full[s]);
            }
            if (w.tmap) {
                for (int64_t y = lo + (int64_t)lane * w.R; y < hi; y += (int64_t)kWarp * w.R)
                    tensor2d_g2s(ring + (y % w.cap) * w.cw, &bmap, col0, (int)y, &full[s]);
            } else if (w.cw == a.N) {
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
        for (int k = max(0, issued - S); k < issued; ++k)
            mbar_wait(&full[k % S], (uint32_t)(k / S) & 1, a.err);
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
    constexpr int kRowBytes = 16 * L;          // one ring row: cw = 4L floats
    const uint32_t ring_a = smem_addr(ring) + 16u * (uint32_t)li;
    const int cap = w.cap;
    const int mask = cap - 1;
    for (int k = 0; k < n_tiles; ++k) {
        const int s = k % S;
        const bool ok = mbar_wait(&full[s], (uint32_t)(k / S) & 1, a.err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int64_t r0 = (t_begin + k) * w.R;
        const int nr = (int)(min(r0 + w.R, a.M) - r0);
        const int s_al = meta[4 * s + 0];
        const bool overflow = meta[4 * s + 1] != 0;
        const int win_lo = meta[4 * s + 2];
        const unsigned win_span = (unsigned)(meta[4 * s + 3] - win_lo);
        const int base = win_lo - win_lo % cap;    // slot(j) = j - base, minus cap if >= cap
        const int *rps = rp + s * w.Rp;
        // shared addresses of entry p: col at cs_a + 4p, val at vs_a + 4p
        const uint32_t cs_a = smem_addr(scol + s * w.ecap) - 4u * (uint32_t)s_al;
        const uint32_t vs_a = smem_addr(sval + s * w.ecap) - 4u * (uint32_t)s_al;

        auto fetch = [&](int j, float (&b)[4]) {
            if (!CHECK || (unsigned)(j - win_lo) < win_span) {
                int slot;
                if constexpr (POW2) {
                    slot = j & mask;
                } else {
                    slot = j - base;
                    if (slot >= cap) slot -= cap;
                }
                lds_v4(ring_a + (uint32_t)slot * kRowBytes, b);
            } else {
                ld_vec<4>(Bg + (int64_t)j * N, b);
            }
        };

        // Entries of one row from the staged segment: batches of 8 independent
        // shared-memory gathers, then 4, then single entries.
        auto run_row = [&](Acc<4, RED, HAS_VAL> &acc, uint32_t ca, uint32_t va, int n) {
            for (; n >= 8; n -= 8, ca += 32, va += 32) {
                int j[8];
                float wv[8], b[8][4];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    j[u] = lds_s32(ca + 4 * u);
                    wv[u] = HAS_VAL ? lds_f32(va + 4 * u) : 1.0f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) fetch(j[u], b[u]);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc.add(wv[u], j[u], b[u]);
            }
            if (n >= 4) {
                int j[4];
                float wv[4], b[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    j[u] = lds_s32(ca + 4 * u);
                    wv[u] = HAS_VAL ? lds_f32(va + 4 * u) : 1.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) fetch(j[u], b[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc.add(wv[u], j[u], b[u]);
                n -= 4;
                ca += 16;
                va += 16;
            }
            for (; n > 0; --n, ca += 4, va += 4) {
                const int j = lds_s32(ca);
                float b[4];
                fetch(j, b);
                acc.add(HAS_VAL ? lds_f32(va) : 1.0f, j, b);
            }
        };
        auto store_row = [&](const Acc<4, RED, HAS_VAL> &acc, int rr, int d) {
            if (!active) return;
            float out[4];
            int arg[4];
            acc.finish(d, out, arg);
            const int64_t i = r0 + rr;
            st_vec<4>(a.C + i * N + c, out);
            if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + i * N + c, arg);
        };

        // Each lane group takes rows grp and grp + kGroups together: two
        // independent entry streams interleaved four entries at a time.
        for (int ra = grp; ra < nr; ra += 2 * kGroups) {
            const int rb = ra + kGroups;
            const int pa = rps[ra], da = rps[ra + 1] - pa;
            const bool has_b = rb < nr;
            const int pb = has_b ? rps[rb] : 0;
            const int db = has_b ? rps[rb + 1] - pb : 0;
            const bool do_a = da <= a.t_split, do_b = has_b && db <= a.t_split;
            Acc<4, RED, HAS_VAL> acc_a, acc_b;
            acc_a.init();
            acc_b.init();
            if (!overflow) {
                uint32_t ca = cs_a + 4u * (uint32_t)pa, va = vs_a + 4u * (uint32_t)pa;
                uint32_t cb = cs_a + 4u * (uint32_t)pb, vb = vs_a + 4u * (uint32_t)pb;
                int na = do_a ? da : 0, nb = do_b ? db : 0;
                for (; na >= 4 && nb >= 4; na -= 4, nb -= 4, ca += 16, va += 16, cb += 16, vb += 16) {
                    int j[8];
                    float wv[8], b[8][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        j[u] = lds_s32(ca + 4 * u);
                        j[4 + u] = lds_s32(cb + 4 * u);
                        wv[u] = HAS_VAL ? lds_f32(va + 4 * u) : 1.0f;
                        wv[4 + u] = HAS_VAL ? lds_f32(vb + 4 * u) : 1.0f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) fetch(j[u], b[u]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc_a.add(wv[u], j[u], b[u]);
#pragma unroll
                    for (int u = 4; u < 8; ++u) acc_b.add(wv[u], j[u], b[u]);
                }
                run_row(acc_a, ca, va, na);
                run_row(acc_b, cb, vb, nb);
            } else {
                for (int q = 0; q < 2; ++q) {
                    const int p0 = q ? pb : pa;
                    const int p1 = p0 + ((q ? do_b : do_a) ? (q ? db : da) : 0);
                    Acc<4, RED, HAS_VAL> &acc = q ? acc_b : acc_a;
                    for (int p = p0; p < p1; ++p) {
                        const int j = ld_stream(a.col + p);
                        float b[4];
                        fetch(j, b);
                        acc.add(HAS_VAL ? ld_stream(a.val + p) : 1.0f, j, b);
                    }
                }
            }
            if (do_a) store_row(acc_a, ra, da);
            if (do_b) store_row(acc_b, rb, db);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

namespace window_detail {
template <int L, int RED, bool HAS_VAL, bool CHECK>
cudaError_t go(const RunArgs &a, const WinShape &w, const CUtensorMap &map, int grid_x, int tiles,
               cudaStream_t s) {
    auto kern = w.pow2 ? k_window<L, RED, HAS_VAL, CHECK, true>
                       : k_window<L, RED, HAS_VAL, CHECK, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         w.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)grid_x, (unsigned)tiles), kWinThreads, w.smem_bytes, s>>>(a, w, map);
    count_launch();
    return cudaGetLastError();
}

template <int RED, bool HAS_VAL, bool CHECK>
cudaError_t by_lanes(const RunArgs &a, const WinShape &w, const CUtensorMap &map, int lanes,
                     int gx, int tiles, cudaStream_t s) {
    switch (lanes) {
        case 2: return go<2, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 4: return go<4, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 8: return go<8, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 16: return go<16, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 32: return go<32, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int RED>
cudaError_t by_flags(const RunArgs &a, const WinShape &w, const CUtensorMap &map, int lanes,
                     bool has_val, bool check, int gx, int tiles, cudaStream_t s) {
    if (has_val)
        return check ? by_lanes<RED, true, true>(a, w, map, lanes, gx, tiles, s)
                     : by_lanes<RED, true, false>(a, w, map, lanes, gx, tiles, s);
    return check ? by_lanes<RED, false, true>(a, w, map, lanes, gx, tiles, s)
                 : by_lanes<RED, false, false>(a, w, map, lanes, gx, tiles, s);
}
}  // namespace window_detail

// Launch of the WINDOW kernel for one reduction (instantiated per reduction in
// f_window_{sum,mean,max}.cu so that the variants compile in parallel).
template <int RED>
cudaError_t launch_window_red(const RunArgs &a, const WinShape &w, const CUtensorMap &map,
                              int lanes, bool has_val, bool check, int gx, int tiles,
                              cudaStream_t s) {
    return window_detail::by_flags<RED>(a, w, map, lanes, has_val, check, gx, tiles, s);
}

extern template cudaError_t launch_window_red<SPMM_SUM>(const RunArgs &, const WinShape &,
                                                        const CUtensorMap &, int, bool, bool,
                                                        int, int, cudaStream_t);
extern template cudaError_t launch_window_red<SPMM_MEAN>(const RunArgs &, const WinShape &,
                                                         const CUtensorMap &, int, bool, bool,
                                                         int, int, cudaStream_t);
extern template cudaError_t launch_window_red<SPMM_MAX>(const RunArgs &, const WinShape &,
                                                        const CUtensorMap &, int, bool, bool,
                                                        int, int, cudaStream_t);

}  // namespace spmm
