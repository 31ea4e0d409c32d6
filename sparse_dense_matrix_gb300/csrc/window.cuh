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
// The producer also writes, per stage, the constants the consumers need for
// the tile (shared addresses of the staged entries, window bounds, ring base).
// Sixteen consumer warps read the entries from shared memory and the gathered
// B rows from the ring. L lanes share a row; each lane owns Q chunks of four
// columns (cw = 4 L Q). With Q = 2, lane groups of even and odd index read
// their two chunks in opposite order, so the two groups that share a
// quarter-warp phase of a 128-bit load touch disjoint halves of their ring
// rows (no bank conflicts when a ring row is 128 bytes), and one slot
// computation serves two 16-byte gathers. An entry outside the window
// (possible only when not every entry is within W) is read from global memory
// instead. Every B row is thus fetched from L2/HBM once per CTA range (plus a
// 2W halo) rather than once per entry.
// Rows longer than t_split are left to the heavy-row split, as everywhere.
// Per lane the entries are accumulated in CSR order with fp32 FMA.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace spmm {

constexpr int kWinMaxStages = 8;
constexpr int kWinConsumerWarps = 16;
constexpr int kWinThreads = (kWinConsumerWarps + 1) * kWarp;
constexpr int kWinMetaInts = 8;   // per-stage constants, see k_window

// shared loads at a compile-time byte offset from a 32-bit shared address
template <int OFF>
__device__ __forceinline__ int lds_s32_at(uint32_t addr) {
    int v;
    asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ float lds_f32_at(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(addr), "n"(OFF));
    return v;
}

// Consumer-side state of one tile and the gathers of a lane.
template <int L, int Q, int RED, bool HAS_VAL, bool CHECK, bool POW2>
struct WinLane {
    using A = Acc<4, RED, HAS_VAL>;
    static constexpr uint32_t kRowBytes = 16u * L * Q;
    uint32_t ring_k[Q];        // shared address of this lane's k-th chunk in ring row 0
    const float *Bg[Q];        // global fallback for out-of-window entries
    int64_t N;
    uint32_t mask, cap;        // ring size (mask = cap - 1 when it is a power of two)
    int win_lo, base;          // tile window start; ring slot of row j = j - base (mod cap)
    unsigned win_span;

    __device__ __forceinline__ void fetch(int j, float (&b)[Q][4]) const {
        if (!CHECK || (unsigned)(j - win_lo) < win_span) {
            uint32_t slot;
            if constexpr (POW2) {
                slot = (uint32_t)j & mask;
            } else {
                const uint32_t s0 = (uint32_t)(j - base);   // in [0, 2 cap)
                slot = min(s0, s0 - cap);                   // s0 or s0 - cap
            }
            const uint32_t ro = slot * kRowBytes;
#pragma unroll
            for (int k = 0; k < Q; ++k) lds_v4(ring_k[k] + ro, b[k]);
        } else {
#pragma unroll
            for (int k = 0; k < Q; ++k) ld_vec<4>(Bg[k] + (int64_t)j * N, b[k]);
        }
    }

    template <int NB, int U = 0>
    __device__ __forceinline__ void load_entries(int (&j)[NB], float (&w)[NB], uint32_t ca,
                                                 uint32_t va) const {
        if constexpr (U < NB) {
            j[U] = lds_s32_at<4 * U>(ca);
            w[U] = HAS_VAL ? lds_f32_at<4 * U>(va) : 1.0f;
            load_entries<NB, U + 1>(j, w, ca, va);
        }
    }

    // NB consecutive entries of one row, all gathers in flight together
    template <int NB>
    __device__ __forceinline__ void run(A (&acc)[Q], uint32_t ca, uint32_t va) const {
        int j[NB];
        float w[NB], b[NB][Q][4];
        load_entries<NB>(j, w, ca, va);
#pragma unroll
        for (int u = 0; u < NB; ++u) fetch(j[u], b[u]);
#pragma unroll
        for (int u = 0; u < NB; ++u)
#pragma unroll
            for (int k = 0; k < Q; ++k) acc[k].add(w[u], j[u], b[u][k]);
    }

    // NB entries of each of two rows, all gathers in flight together
    template <int NB>
    __device__ __forceinline__ void run2(A (&aa)[Q], uint32_t ca, uint32_t va, A (&ab)[Q],
                                         uint32_t cb, uint32_t vb) const {
        int j[2 * NB];
        float w[2 * NB], b[2 * NB][Q][4];
        int (&ja)[NB] = *reinterpret_cast<int (*)[NB]>(&j[0]);
        int (&jb)[NB] = *reinterpret_cast<int (*)[NB]>(&j[NB]);
        float (&wa)[NB] = *reinterpret_cast<float (*)[NB]>(&w[0]);
        float (&wb)[NB] = *reinterpret_cast<float (*)[NB]>(&w[NB]);
        load_entries<NB>(ja, wa, ca, va);
        load_entries<NB>(jb, wb, cb, vb);
#pragma unroll
        for (int u = 0; u < 2 * NB; ++u) fetch(j[u], b[u]);
#pragma unroll
        for (int u = 0; u < NB; ++u)
#pragma unroll
            for (int k = 0; k < Q; ++k) aa[k].add(w[u], j[u], b[u][k]);
#pragma unroll
        for (int u = NB; u < 2 * NB; ++u)
#pragma unroll
            for (int k = 0; k < Q; ++k) ab[k].add(w[u], j[u], b[u][k]);
    }

    // the n entries of one row: batches of 8 / Q gathered rows (8 16-byte
    // gathers in flight per lane), then 4, 2 and 1
    __device__ __forceinline__ void run_row(A (&acc)[Q], uint32_t ca, uint32_t va, int n) const {
        if constexpr (Q == 1) {
            for (; n >= 8; n -= 8, ca += 32, va += 32) run<8>(acc, ca, va);
            if (n >= 4) {
                run<4>(acc, ca, va);
                n -= 4; ca += 16; va += 16;
            }
        } else {
            for (; n >= 4; n -= 4, ca += 16, va += 16) run<4>(acc, ca, va);
        }
        if (n >= 2) {
            run<2>(acc, ca, va);
            n -= 2; ca += 8; va += 8;
        }
        if (n) run<1>(acc, ca, va);
    }
};

// EPI: the fused bias/ReLU epilogue is compiled in only where it is used
template <int L, int Q, int RED, bool HAS_VAL, bool CHECK, bool POW2, bool EPI>
__global__ void __launch_bounds__(kWinThreads, 1)
    k_window(const RunArgs a, const WinShape w, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 128-byte aligned base (tensor copies want 128-byte aligned destinations)
    unsigned char *smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kWinMaxStages;
    const int S = w.S;
    int *meta = reinterpret_cast<int *>(smem + w.off_meta);      // [S][kWinMetaInts]
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
        // This warp shares its scheduler with four consumer warps and must issue
        // a tile's copies well before the consumers reach it, so the per-tile
        // bookkeeping is done 32 tiles at a time: lane l works out tile kb + l
        // (segment bounds, window, the new ring rows and their slot), and the
        // serial loop over the tiles only reads those values by shuffles.
        const int64_t R = w.R, W = w.W;
        const int64_t Kr = (a.K + R - 1) / R * R;   // B rows rounded up to whole boxes
        const uint32_t cap = (uint32_t)w.cap;
        // row-pointer values of a batch, loaded one batch ahead
        auto seg_load = [&](int kk, int &b, int &e) {
            const int64_t q0 = min((t_begin + kk) * R, a.M);
            b = ld_stream(a.rowptr + q0);
            e = ld_stream(a.rowptr + min(q0 + R, a.M));
        };
        int nb_b, nb_e;
        seg_load(min(lane, n_tiles), nb_b, nb_e);
        int64_t carry_hi = -1;   // highest B row requested before this batch (+1)
        int s = 0;
        uint32_t round = 0;      // tile / S
        int issued = 0;
        bool failed = false;
        for (int kb = 0; kb < n_tiles && !failed; kb += kWarp) {
            // ---- this lane's tile: kb + lane
            const int kt = kb + lane;
            const int seg_b = nb_b, seg_e = nb_e;
            if (kb + kWarp < n_tiles) seg_load(min(kb + kWarp + lane, n_tiles), nb_b, nb_e);
            const int64_t r0 = (t_begin + kt) * R;
            const int64_t r1 = min(r0 + R, a.M);
            const int s_al = seg_b & ~3;
            const bool overflow = (seg_e - s_al) > w.ecap;
            const int e_cp = overflow ? s_al : max(s_al, min((seg_e + 3) & ~3, a.nnz4));
            // window of the tile around its global rows [g0, g1) (a row-range
            // plan's local row 0 is global row a.row0, a multiple of R); empty
            // when it lies past the last B row
            const int64_t g0 = r0 + a.row0, g1 = r1 + a.row0;
            const int64_t win_lo = max(g0 - W, (int64_t)0);
            const int64_t win_hi = max(min(g1 + W, a.K), win_lo);
            // rows requested through this tile: whole R-row boxes when the ring
            // holds a column slice (W and the tile starts are multiples of R);
            // non-decreasing in the tile index
            const int64_t top = w.tmap ? min(g0 + R + W, Kr) : win_hi;
            int64_t prev = __shfl_up_sync(0xffffffffu, top, 1);
            if (lane == 0) prev = carry_hi;
            carry_hi = __shfl_sync(0xffffffffu, top, kWarp - 1);
            // new rows [lo, hi): contiguous with what is loaded
            const int64_t lo = (prev >= win_lo) ? prev : win_lo;
            const int64_t hi = max(top, lo);
            const uint32_t lo_slot = (uint32_t)(lo % cap);
            const uint32_t win_mod = (uint32_t)(win_lo % cap);
            const int t_n_new = (int)(hi - lo);            // <= R + 2W <= cap
            const int t_lo = (int)lo, t_win_lo = (int)win_lo, t_span = (int)(win_hi - win_lo);
            const int t_base = (int)(win_lo - win_mod);

            const int n_here = min(kWarp, n_tiles - kb);
            for (int t = 0; t < n_here; ++t) {
                const int k = kb + t;
                if (round > 0) {
                    const bool ok = mbar_wait(&empty[s], (round - 1) & 1, a.err);
                    if (!__all_sync(0xffffffffu, ok)) {
                        failed = true;
                        break;
                    }
                }
                const int c_sal = __shfl_sync(0xffffffffu, s_al, t);
                const int c_ecp = __shfl_sync(0xffffffffu, e_cp, t);
                const int c_sege = __shfl_sync(0xffffffffu, seg_e, t);
                const bool c_over = __shfl_sync(0xffffffffu, overflow ? 1 : 0, t) != 0;
                const int c_lo = __shfl_sync(0xffffffffu, t_lo, t);
                const uint32_t c_slot = __shfl_sync(0xffffffffu, lo_slot, t);
                const uint32_t c_new = (uint32_t)__shfl_sync(0xffffffffu, t_n_new, t);
                const int64_t c_r0 = (t_begin + k) * R;
                int *rps = rp + s * w.Rp;
                int *scs = scol + s * w.ecap;
                float *svs = sval + s * w.ecap;
                // the last < 4 entries of the whole array: plain loads
                if (!c_over) {
                    for (int p = c_ecp + lane; p < c_sege; p += kWarp) {
                        scs[p - c_sal] = ld_stream(a.col + p);
                        if (HAS_VAL) svs[p - c_sal] = ld_stream(a.val + p);
                    }
                }
                const int c_wlo = __shfl_sync(0xffffffffu, t_win_lo, t);
                const int c_span = __shfl_sync(0xffffffffu, t_span, t);
                const int c_base = __shfl_sync(0xffffffffu, t_base, t);
                if (lane == 0) {
                    // constants of the tile for the consumers (published by the
                    // arrive below, which orders these stores before the phase flip)
                    int *m = meta + kWinMetaInts * s;
                    m[0] = (int)(smem_addr(scs) - 4u * (uint32_t)c_sal);
                    m[1] = (int)(smem_addr(svs) - 4u * (uint32_t)c_sal);
                    m[2] = c_over ? 1 : 0;
                    m[3] = c_wlo;
                    m[4] = c_span;
                    m[5] = c_base;
                }
                const uint32_t ring_bytes = c_new * (uint32_t)(w.tmap ? w.cw : cw_eff) * 4u;
                const uint32_t seg_bytes = (uint32_t)(c_ecp - c_sal) * 4u;
                const uint32_t rp_bytes = (uint32_t)w.Rp * 4u;
                const uint32_t tx = rp_bytes + seg_bytes * (HAS_VAL ? 2u : 1u) + ring_bytes;
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&full[s], tx);
                __syncwarp();
                // row pointers of the tile: the plan's copy is padded past rowptr[M]
                if (lane == 3) bulk_g2s(rps, a.rowptr + c_r0, rp_bytes, &full[s]);
                if (seg_bytes) {
                    if (lane == 0) bulk_g2s(scs, a.col + c_sal, seg_bytes, &full[s]);
                    if (HAS_VAL && lane == 1) bulk_g2s(svs, a.val + c_sal, seg_bytes, &full[s]);
                }
                if (w.tmap) {
                    // boxes of R rows start on multiples of R and never wrap (cap is one)
                    for (uint32_t d = (uint32_t)lane * (uint32_t)R; d < c_new;
                         d += kWarp * (uint32_t)R) {
                        uint32_t slot = c_slot + d;
                        if (slot >= cap) slot -= cap;
                        tensor2d_g2s(ring + (size_t)slot * w.cw, &bmap, col0, c_lo + (int)d,
                                     &full[s]);
                    }
                } else if (w.cw == a.N) {
                    // ring rows are whole B rows: one copy per run up to the ring's wrap
                    if (lane == 2) {
                        uint32_t d = 0, slot = c_slot;
                        while (d < c_new) {
                            const uint32_t run = min(c_new - d, cap - slot);
                            bulk_g2s(ring + (size_t)slot * w.cw, a.B + ((int64_t)c_lo + d) * N,
                                     run * (uint32_t)N * 4u, &full[s]);
                            d += run;
                            slot += run;
                            if (slot >= cap) slot -= cap;
                        }
                    }
                } else {
                    for (uint32_t d = (uint32_t)lane; d < c_new; d += kWarp) {
                        uint32_t slot = c_slot + d;
                        if (slot >= cap) slot -= cap;
                        bulk_g2s(ring + (size_t)slot * w.cw, a.B + ((int64_t)c_lo + d) * N + col0,
                                 (uint32_t)cw_eff * 4u, &full[s]);
                    }
                }
                issued = k + 1;
                if (++s == S) {
                    s = 0;
                    ++round;
                }
            }
        }
        // never leave while copies this warp issued may still be landing
        for (int k = max(0, issued - S); k < issued; ++k)
            mbar_wait(&full[k % S], (uint32_t)(k / S) & 1, a.err);
        return;
    }

    // -------------------------------------------------------------- consumers
    using Lane = WinLane<L, Q, RED, HAS_VAL, CHECK, POW2>;
    using A = typename Lane::A;
    constexpr int kGroups = kWinConsumerWarps * kWarp / L;
    const int ct = threadIdx.x - kWarp;
    const int grp = ct / L;
    const int li = ct % L;
    const int rot = Q > 1 ? grp % Q : 0;
    Lane ln;
    int cq[Q];                                   // first column of each chunk
    bool act[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        const int chunk = li + L * ((k + rot) % Q);
        ln.ring_k[k] = smem_addr(ring) + 16u * (uint32_t)chunk;
        cq[k] = col0 + 4 * chunk;
        act[k] = cq[k] < a.N;
        ln.Bg[k] = a.B + min(cq[k], a.N - 4);    // clamped for idle lanes
    }
    ln.N = N;
    ln.cap = (uint32_t)w.cap;
    ln.mask = (uint32_t)w.cap - 1u;

    int64_t t_r0 = t_begin * w.R;               // first row of the current tile
    auto store_row = [&](const A (&acc)[Q], int rr, int d) {
        const int64_t i = t_r0 + rr;
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            if (!act[k]) continue;
            float out[4];
            int arg[4];
            acc[k].finish(d, out, arg);
            if constexpr (EPI) epilogue<4>(a, cq[k], out);
            st_vec<4>(a.C + i * N + cq[k], out);
            if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + i * N + cq[k], arg);
        }
    };

    int s = 0;
    uint32_t phase = 0;
    for (int k = 0; k < n_tiles; ++k, t_r0 += w.R) {
        const bool ok = mbar_wait(&full[s], phase, a.err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int nr = (int)(min(t_r0 + w.R, a.M) - t_r0);
        const int *m = meta + kWinMetaInts * s;
        const uint32_t cs_a = (uint32_t)m[0];   // shared address of entry p: cs_a + 4p
        const uint32_t vs_a = (uint32_t)m[1];
        const bool overflow = m[2] != 0;
        ln.win_lo = m[3];
        ln.win_span = (unsigned)m[4];
        ln.base = m[5];
        const int *rps = rp + s * w.Rp;

        // Each lane group takes rows grp and grp + kGroups together: two
        // independent entry streams interleaved four entries at a time.
        for (int ra = grp; ra < nr; ra += 2 * kGroups) {
            const int rb = ra + kGroups;
            const int pa = rps[ra], da = rps[ra + 1] - pa;
            const bool has_b = rb < nr;
            const int pb = has_b ? rps[rb] : 0;
            const int db = has_b ? rps[rb + 1] - pb : 0;
            const bool do_a = da <= a.t_split, do_b = has_b && db <= a.t_split;
            A acc_a[Q], acc_b[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                acc_a[q].init();
                acc_b[q].init();
            }
            if (!overflow) {
                uint32_t ca = cs_a + 4u * (uint32_t)pa, va = vs_a + 4u * (uint32_t)pa;
                uint32_t cb = cs_a + 4u * (uint32_t)pb, vb = vs_a + 4u * (uint32_t)pb;
                int na = do_a ? da : 0, nb = do_b ? db : 0;
                constexpr int kPair = 4 / Q;   // entries per row per step of the pair loop
                for (; na >= kPair && nb >= kPair; na -= kPair, nb -= kPair, ca += 4 * kPair,
                                                   va += 4 * kPair, cb += 4 * kPair, vb += 4 * kPair)
                    ln.template run2<kPair>(acc_a, ca, va, acc_b, cb, vb);
                ln.run_row(acc_a, ca, va, na);
                if (nb) ln.run_row(acc_b, cb, vb, nb);
            } else {
                for (int q = 0; q < 2; ++q) {
                    const int p0 = q ? pb : pa;
                    const int p1 = p0 + ((q ? do_b : do_a) ? (q ? db : da) : 0);
                    A (&acc)[Q] = q ? acc_b : acc_a;
                    for (int p = p0; p < p1; ++p) {
                        const int j = ld_stream(a.col + p);
                        const float wv = HAS_VAL ? ld_stream(a.val + p) : 1.0f;
                        float b[Q][4];
                        ln.fetch(j, b);
#pragma unroll
                        for (int kk = 0; kk < Q; ++kk) acc[kk].add(wv, j, b[kk]);
                    }
                }
            }
            if (do_a) store_row(acc_a, ra, da);
            if (do_b) store_row(acc_b, rb, db);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == S) {
            s = 0;
            phase ^= 1u;
        }
    }
}

namespace window_detail {
template <int L, int Q, int RED, bool HAS_VAL, bool CHECK>
cudaError_t go(const RunArgs &a, const WinShape &w, const CUtensorMap &map, int grid_x, int tiles,
               cudaStream_t s) {
    const bool epi = a.bias != nullptr || a.act != SPMM_ACT_NONE;
    auto kern = w.pow2 ? (epi ? k_window<L, Q, RED, HAS_VAL, CHECK, true, true>
                              : k_window<L, Q, RED, HAS_VAL, CHECK, true, false>)
                       : (epi ? k_window<L, Q, RED, HAS_VAL, CHECK, false, true>
                              : k_window<L, Q, RED, HAS_VAL, CHECK, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         w.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)grid_x, (unsigned)tiles), kWinThreads, w.smem_bytes, s>>>(a, w, map);
    count_launch();
    return cudaGetLastError();
}

// (L, Q) shapes: column tiles of 8 (2 x 1), 16 (2 x 2), 32 (4 x 2), 64 (8 x 2)
// and 128 (16 x 2) columns
template <int RED, bool HAS_VAL, bool CHECK>
cudaError_t by_lanes(const RunArgs &a, const WinShape &w, const CUtensorMap &map, int gx,
                     int tiles, cudaStream_t s) {
    const int key = w.L * 4 + w.Q;
    switch (key) {
        case 2 * 4 + 1: return go<2, 1, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 2 * 4 + 2: return go<2, 2, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 4 * 4 + 1: return go<4, 1, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 4 * 4 + 2: return go<4, 2, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 8 * 4 + 2: return go<8, 2, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        case 16 * 4 + 2: return go<16, 2, RED, HAS_VAL, CHECK>(a, w, map, gx, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int RED>
cudaError_t by_flags(const RunArgs &a, const WinShape &w, const CUtensorMap &map, bool has_val,
                     bool check, int gx, int tiles, cudaStream_t s) {
    if (has_val)
        return check ? by_lanes<RED, true, true>(a, w, map, gx, tiles, s)
                     : by_lanes<RED, true, false>(a, w, map, gx, tiles, s);
    return check ? by_lanes<RED, false, true>(a, w, map, gx, tiles, s)
                 : by_lanes<RED, false, false>(a, w, map, gx, tiles, s);
}
}  // namespace window_detail

// Launch of the WINDOW kernel for one reduction (instantiated per reduction in
// f_window_{sum,mean,max}.cu so that the variants compile in parallel).
template <int RED>
cudaError_t launch_window_red(const RunArgs &a, const WinShape &w, const CUtensorMap &map,
                              bool has_val, bool check, int gx, int tiles, cudaStream_t s) {
    return window_detail::by_flags<RED>(a, w, map, has_val, check, gx, tiles, s);
}

extern template cudaError_t launch_window_red<SPMM_SUM>(const RunArgs &, const WinShape &,
                                                        const CUtensorMap &, bool, bool, int,
                                                        int, cudaStream_t);
extern template cudaError_t launch_window_red<SPMM_MEAN>(const RunArgs &, const WinShape &,
                                                         const CUtensorMap &, bool, bool, int,
                                                         int, cudaStream_t);
extern template cudaError_t launch_window_red<SPMM_MAX>(const RunArgs &, const WinShape &,
                                                        const CUtensorMap &, bool, bool, int,
                                                        int, cudaStream_t);

}  // namespace spmm
