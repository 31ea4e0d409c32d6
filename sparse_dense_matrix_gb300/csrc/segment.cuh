// SEGMENT family: entry-balanced merge-path tiles for skewed (power-law)
// graphs whose column ids carry no locality.
//
// The CSR traversal is cut into tiles of kSegItems items, an item being one
// stored entry or one row end, along the merge path of the row ends
// (rowptr[1..M]) with the entry indices (0..nnz-1). Tile t starts at item
// k = t * kSegItems, after r_t row ends and e_t = k - r_t entries, where r_t is
// the number of rows i >= 1 with rowptr[i] + i <= k; the plan holds (r_t, e_t)
// for every tile. Every tile carries the same work whatever the degree
// distribution: a hub row of 1e5 entries spans many tiles, and a run of empty
// rows costs one item per row (ParamSpMM section 3.2, nonzero-split workload
// balancing; graph-spmm card, "Requirements and limits": hubs want a
// segmented schedule).
//
// Each warp of a persistent grid owns a contiguous range of tiles and is its
// own producer: lane 0 copies a tile's row pointers, columns and values into a
// private shared-memory stage with 1-D bulk copies (cp.async.bulk completing
// on the stage's mbarrier), one tile ahead of the tile being reduced,
// so the dependent rowptr -> col chain never waits on DRAM and only the
// gathers of B rows are exposed. Within a tile, the G = 32 / L lane groups of
// the warp take equal slices of the items (a second merge-path search, over
// the staged row pointers). A group walks its slice in batches of U entries,
// with all U gathers (128-bit, through L1) in flight together, and crosses row
// ends inside a batch: a row that begins and ends in the slice is finished and
// stored at once. The partial rows at the slices' edges are combined in slice
// order through warp shuffles, and a row still open at the end of a tile is
// carried in registers into the next tile. Only the rows open at the two ends
// of a warp's tile range leave the kernel as partials; a second launch
// combines those in warp order and stores them. Every summation order is a
// pure function of the plan, N and the grid: no atomics, bitwise
// reproducible (DualGCN section 3.3: several independent gathers in flight
// per lane).
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace spmm {

// Two stages: a third (213 KB of shared memory per SM instead of 142 KB)
// leaves the L1 cache too small for the hub rows of B, and measured 1.8x
// slower on the 4M-row Chung-Lu graph at N = 16.
#ifndef SPMM_SEG_STAGES
#define SPMM_SEG_STAGES 2
#endif
#ifndef SPMM_SEG_BATCH
#define SPMM_SEG_BATCH 8
#endif
constexpr int kSegStages = SPMM_SEG_STAGES;
constexpr int kSegThreads = kSegWarps * kWarp;
constexpr int kSegRegionA = kSegItems + 16;   // row pointers, then columns (ints)
constexpr int kSegRegionV = kSegItems + 8;    // values
constexpr int kSegStageInts = kSegRegionA + kSegRegionV;
constexpr int kSegBarBytes = kSegWarps * kSegStages * 8;
constexpr int kSegSmemBytes = kSegBarBytes + kSegWarps * kSegStages * kSegStageInts * 4;
static_assert(kSegBarBytes % 16 == 0 && (kSegStageInts * 4) % 16 == 0, "16-byte stages");
static_assert(kSegItems % 16 == 0, "slices of whole items for up to 16 lane groups");

// x := x (+) y: the sum in this order, or the (value, column) maximum
template <int RED, bool HV>
__device__ __forceinline__ void seg_merge(Acc<4, RED, HV> &x, const float (&v)[4],
                                          const int (&j)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if constexpr (RED == SPMM_MAX) {
            if (max_better(v[e], j[e], x.v[e], x.j[e])) { x.v[e] = v[e]; x.j[e] = j[e]; }
        } else {
            x.v[e] = __fadd_rn(x.v[e], v[e]);
        }
    }
}

template <int L, int Q, int RED, bool HAS_VAL, bool EPI>
__global__ void __launch_bounds__(kSegThreads, 1) k_segment(const RunArgs a) {
    constexpr int G = kWarp / L;               // lane groups per warp
    constexpr int SLICE = kSegItems / G;       // items per group slice
    constexpr int U = (Q == 1) ? SPMM_SEG_BATCH : (RED == SPMM_MAX ? 2 : 4);   // entries per batch
    constexpr int CW = 4 * L * Q;              // columns of one column tile
    constexpr unsigned FULL = 0xffffffffu;
    using A = Acc<4, RED, HAS_VAL>;

    extern __shared__ __align__(16) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    int *stages = reinterpret_cast<int *>(smem + kSegBarBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & (kWarp - 1);
    const int g = lane / L, t = lane % L;
    uint64_t *bar = bars + warp * kSegStages;
    if (lane == 0) {
        for (int s = 0; s < kSegStages; ++s) mbar_init(&bar[s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    const int W = a.seg_warps;
    const int wg = blockIdx.x * kSegWarps + warp;
    if (wg >= W) return;                       // uniform per warp
    const int64_t n = a.seg_n_tiles;
    const int64_t t0 = n * wg / W;
    const int nt = (int)(n * (wg + 1) / W - t0);
    int *stage = stages + (size_t)warp * kSegStages * kSegStageInts;
    const int64_t N = a.N;

    // this lane's columns: Q chunks of four, col0 + 4 (t + L q)
    const int col0 = blockIdx.y * CW;
    int cq[Q];
    bool act[Q];
    const float *Bq[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        cq[q] = col0 + 4 * (t + L * q);
        act[q] = cq[q] < a.N;
        Bq[q] = a.B + min(cq[q], a.N - 4);     // clamped for idle lanes
    }

    // Tile table: lane l holds the (rows ended, entries consumed) pair of tile
    // t0 + 32 b + l for the batch b = tb_base (cur) and the next one; the issue
    // point needs at most four tiles past the one being reduced.
    auto tbl_load = [&](int b) -> int2 {
        const int64_t idx = min(t0 + 32 * (int64_t)b + lane, n);
        return a.seg_tiles[idx];
    };
    int2 tb_cur = tbl_load(0), tb_next = tbl_load(1);
    int tb_base = 0;
    auto tile_at = [&](int i) -> int2 {        // uniform i in [32 tb_base, 32 tb_base + 64)
        const int rel = i - 32 * tb_base;
        const int src = rel & 31;
        const int cx = __shfl_sync(FULL, tb_cur.x, src), cy = __shfl_sync(FULL, tb_cur.y, src);
        const int nx = __shfl_sync(FULL, tb_next.x, src), ny = __shfl_sync(FULL, tb_next.y, src);
        return rel < 32 ? make_int2(cx, cy) : make_int2(nx, ny);
    };

    // Bulk copies of tile i into stage s: row pointers [r_t & ~3, ...) up to
    // rowptr[r_{t+1} + 1], then the columns [e_t & ~3, ...) up to e_{t+1}
    // (both rounded to whole 16-byte words; the plan's rowptr is padded), and
    // the values. The last (< 4) entries of the whole array come by plain loads.
    auto issue = [&](int i, int s) {
        const int2 p = tile_at(i), q = tile_at(i + 1);
        const int rb0 = p.x & ~3;
        const int rcnt = ((q.x + 2 + 3) & ~3) - rb0;
        const int eb0 = p.y & ~3;
        const int eend = min((q.y + 3) & ~3, a.nnz4);
        const int ecnt = max(0, eend - eb0);
        int *st = stage + s * kSegStageInts;
        int *cs = st + rcnt;
        float *vs = reinterpret_cast<float *>(st + kSegRegionA);
        for (int e = max(eend, eb0) + lane; e < q.y; e += kWarp) {
            cs[e - eb0] = ld_stream(a.col + e);
            if (HAS_VAL) vs[e - eb0] = ld_stream(a.val + e);
        }
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_shared();
            const uint32_t bytes = (uint32_t)rcnt * 4u + (uint32_t)ecnt * (HAS_VAL ? 8u : 4u);
            mbar_arrive_expect_tx(&bar[s], bytes);
            bulk_g2s(st, a.rowptr + rb0, (uint32_t)rcnt * 4u, &bar[s]);
            if (ecnt) {
                bulk_g2s(cs, a.col + eb0, (uint32_t)ecnt * 4u, &bar[s]);
                if (HAS_VAL) bulk_g2s(vs, a.val + eb0, (uint32_t)ecnt * 4u, &bar[s]);
            }
        }
        __syncwarp();
    };

    // the finished row `row` of d entries from accumulators x (by this lane's columns)
    auto store_row = [&](int64_t row, const A (&x)[Q], int d) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (!act[q]) continue;
            float out[4];
            int arg[4];
            x[q].finish(d, out, arg);
            if constexpr (RED == SPMM_SUM) mean_scale<4>(a, d, out);
            if constexpr (EPI) epilogue<4>(a, cq[q], out);
            st_vec<4>(a.C + row * N + cq[q], out);
            if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + row * N + cq[q], arg);
        }
    };
    // an open row's partial to slot (0: the row open at the start of the warp's
    // range, 1: the row open at its end)
    auto store_carry = [&](int slot, const A (&x)[Q]) {
        const int64_t base = (((int64_t)blockIdx.y * W + wg) * 2 + slot) * CW;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (!act[q]) continue;
            const int64_t o = base + 4 * (t + L * q);
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = x[q].v[e];
            st_vec<4>(a.seg_cval + o, v);
            if constexpr (RED == SPMM_MAX) st_vec_i<4>(a.seg_carg + o, x[q].j);
        }
    };

    // the row open across tiles: mode 0 none, 1 began in this warp's range,
    // 2 began before it (its result leaves as the range's head partial)
    A cur[Q];
    int cur_row = -1, cur_mode = 0;
    int h0_row = -1, h0_ends = 0, tail_row = -1;

    const int pre = min(nt, kSegStages);
    for (int i = 0; i < pre; ++i) issue(i, i);
    int issued = pre;
    bool failed = false;

    for (int i = 0; i < nt; ++i) {
        if (i >= 32 * (tb_base + 1)) {         // next batch of the tile table
            tb_cur = tb_next;
            ++tb_base;
            tb_next = tbl_load(tb_base + 1);
        }
        const int s = i % kSegStages;
        const bool ok = mbar_wait(&bar[s], (uint32_t)(i / kSegStages) & 1u, a.err);
        if (!__all_sync(FULL, ok)) {
            failed = true;
            break;
        }
        const int2 p = tile_at(i), q = tile_at(i + 1);
        const int rb0 = p.x & ~3, eb0 = p.y & ~3;
        const int rcnt = ((q.x + 2 + 3) & ~3) - rb0;
        const int *st = stage + s * kSegStageInts;
        const int *rps = st - rb0;             // rps[r] = rowptr[r] for the tile's rows
        const int *cs = st + rcnt - eb0;       // cs[e] = col[e] for the tile's entries
        const float *vs = reinterpret_cast<const float *>(st + kSegRegionA) - eb0;

        // ---- this group's slice [ka, kb) of the tile's items
        const int64_t kend = (int64_t)q.x + q.y;
        const int64_t ka = min((t0 + i) * (int64_t)kSegItems + (int64_t)g * SLICE, kend);
        int lo = p.x, hi = q.x;                // largest r with rowptr[r] + r <= ka
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)rps[mid] + mid <= ka) lo = mid;
            else hi = mid - 1;
        }
        const int ra = lo, ea = (int)(ka - ra);
        int rb = __shfl_down_sync(FULL, ra, L), eb = __shfl_down_sync(FULL, ea, L);
        if (g == G - 1) { rb = q.x; eb = q.y; }
        const bool nonempty = ra < rb || ea < eb;
        // the slice's first row began before the slice: its part is a head record
        const int r_before = (nonempty && rps[ra] < ea) ? ra : -1;

        A acc[Q], hrec[Q], trec[Q];
#pragma unroll
        for (int qq = 0; qq < Q; ++qq) {
            acc[qq].init();
            hrec[qq].init();
            trec[qq].init();
        }
        int h_ends = 0, t_row = -1;
        int r = ra;
        int rend = rps[r + 1];
        bool touched = false;
        auto emit = [&](int row) {             // row ends here
            if (row == r_before) {
#pragma unroll
                for (int qq = 0; qq < Q; ++qq) hrec[qq] = acc[qq];
                h_ends = 1;
            } else {
                store_row(row, acc, rps[row + 1] - rps[row]);
            }
        };
        for (int e = ea; e < eb; e += U) {
            const int nb = min(U, eb - e);
            int j[U];
            float w[U], b[U][Q][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool in = u < nb;
                j[u] = in ? cs[e + u] : 0;
                w[u] = (HAS_VAL && in) ? vs[e + u] : 1.0f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u < nb) {
#pragma unroll
                    for (int qq = 0; qq < Q; ++qq) ld_vec<4>(Bq[qq] + (int64_t)j[u] * N, b[u][qq]);
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u < nb) {
                    while (e + u >= rend) {
                        emit(r);
                        ++r;
                        rend = rps[r + 1];
#pragma unroll
                        for (int qq = 0; qq < Q; ++qq) acc[qq].init();
                        touched = false;
                    }
#pragma unroll
                    for (int qq = 0; qq < Q; ++qq) acc[qq].add(w[u], j[u], b[u][qq]);
                    touched = true;
                }
        }
        for (; r < rb; ++r) {                  // the row ends left in the slice
            emit(r);
#pragma unroll
            for (int qq = 0; qq < Q; ++qq) acc[qq].init();
            touched = false;
        }
        if (touched) {                         // row rb continues past the slice
            if (r == r_before) {
#pragma unroll
                for (int qq = 0; qq < Q; ++qq) hrec[qq] = acc[qq];
                h_ends = 0;
            } else {
#pragma unroll
                for (int qq = 0; qq < Q; ++qq) trec[qq] = acc[qq];
                t_row = r;
            }
        }

        // ---- combine the slices' edge records in slice order (uniform loop)
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            const int src0 = gg * L;
            const int hr = __shfl_sync(FULL, r_before, src0);
            const int he = __shfl_sync(FULL, h_ends, src0);
            const int tr = __shfl_sync(FULL, t_row, src0);
            if (hr >= 0) {
                if (cur_mode == 0) {           // the row open at the start of the range
#pragma unroll
                    for (int qq = 0; qq < Q; ++qq) cur[qq].init();
                    cur_row = hr;
                    cur_mode = 2;
                    h0_row = hr;
                }
#pragma unroll
                for (int qq = 0; qq < Q; ++qq) {
                    float hv[4];
                    int hj[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hv[e] = __shfl_sync(FULL, hrec[qq].v[e], src0 + t);
                        hj[e] = RED == SPMM_MAX ? __shfl_sync(FULL, hrec[qq].j[e], src0 + t) : 0;
                    }
                    seg_merge<RED, HAS_VAL>(cur[qq], hv, hj);
                }
                if (he) {
                    if (cur_mode == 1) {
                        if (g == 0) store_row(cur_row, cur, rps[cur_row + 1] - rps[cur_row]);
                    } else {
                        if (g == 0) store_carry(0, cur);
                        h0_ends = 1;
                    }
                    cur_mode = 0;
                }
            }
            if (tr >= 0) {
#pragma unroll
                for (int qq = 0; qq < Q; ++qq)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        cur[qq].v[e] = __shfl_sync(FULL, trec[qq].v[e], src0 + t);
                        if constexpr (RED == SPMM_MAX)
                            cur[qq].j[e] = __shfl_sync(FULL, trec[qq].j[e], src0 + t);
                    }
                cur_row = tr;
                cur_mode = 1;
            }
        }
        __syncwarp();
        if (issued < nt) {                     // this stage is free again
            issue(issued, s);
            ++issued;
        }
    }
    if (!failed) {
        if (cur_mode == 1) {
            if (g == 0) store_carry(1, cur);
            tail_row = cur_row;
        } else if (cur_mode == 2) {
            if (g == 0) store_carry(0, cur);
            h0_ends = 0;
        }
        if (lane == 0 && blockIdx.y == 0) a.seg_meta[wg] = make_int4(h0_row, h0_ends, tail_row, 0);
    } else {
        // never leave while copies this warp issued may still be landing
        for (int k = max(0, issued - kSegStages); k < issued; ++k)
            mbar_wait(&bar[k % kSegStages], (uint32_t)(k / kSegStages) & 1u, a.err);
    }
}

// The rows left open at the ends of the warps' tile ranges: the tail partial of
// warp w, then the head partials of warps w + 1, w + 2, ... in order until the
// row ends; one thread per (warp range, four columns).
template <int RED>
__global__ void __launch_bounds__(256) k_segment_fix(const RunArgs a, int cw) {
    const int n_vec = a.N / 4;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int W = a.seg_warps;
    if (idx >= (int64_t)W * n_vec) return;
    const int w = (int)(idx / n_vec), vi = (int)(idx % n_vec);
    const int4 m = a.seg_meta[w];
    const int r = m.z;
    if (r < 0) return;
    const int y = vi * 4 / cw, off = vi * 4 - y * cw;
    auto slot = [&](int ww, int sl) { return (((int64_t)y * W + ww) * 2 + sl) * cw + off; };
    float v[4];
    int j[4] = {0, 0, 0, 0};
    ld_vec<4>(a.seg_cval + slot(w, 1), v);
    if constexpr (RED == SPMM_MAX) {
        const int4 q = __ldg(reinterpret_cast<const int4 *>(a.seg_carg + slot(w, 1)));
        j[0] = q.x; j[1] = q.y; j[2] = q.z; j[3] = q.w;
    }
    for (int u = w + 1; u < W; ++u) {
        const int4 mu = a.seg_meta[u];
        float x[4];
        ld_vec<4>(a.seg_cval + slot(u, 0), x);
        if constexpr (RED == SPMM_MAX) {
            const int4 q = __ldg(reinterpret_cast<const int4 *>(a.seg_carg + slot(u, 0)));
            const int xj[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (max_better(x[e], xj[e], v[e], j[e])) { v[e] = x[e]; j[e] = xj[e]; }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = __fadd_rn(v[e], x[e]);
        }
        if (mu.y) break;
    }
    const int d = a.rowptr[r + 1] - a.rowptr[r];
    const int64_t c = (int64_t)vi * 4;
    float out[4];
    int arg[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if constexpr (RED == SPMM_MAX) {
            const bool none = j[e] == kNoCol;
            out[e] = none ? 0.0f : v[e];
            arg[e] = none ? -1 : j[e];
        } else {
            out[e] = v[e];
            arg[e] = 0;
        }
    }
    if constexpr (RED == SPMM_SUM) mean_scale<4>(a, d, out);
    epilogue<4>(a, c, out);
    st_vec<4>(a.C + (int64_t)r * a.N + c, out);
    if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + (int64_t)r * a.N + c, arg);
}

namespace segment_detail {
template <int L, int Q, int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, int ctas_x, int tiles_y, cudaStream_t s) {
    const bool epi = a.bias != nullptr || a.act != SPMM_ACT_NONE;
    auto kern = epi ? k_segment<L, Q, RED, HAS_VAL, true> : k_segment<L, Q, RED, HAS_VAL, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSegSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)ctas_x, (unsigned)tiles_y), kSegThreads, kSegSmemBytes, s>>>(a);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = (int64_t)a.seg_warps * (a.N / 4);
    k_segment_fix<RED><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a, 4 * L * Q);
    count_launch();
    return cudaGetLastError();
}

template <int RED, bool HAS_VAL>
cudaError_t by_shape(const RunArgs &a, int lanes, int chunks, int ctas_x, int tiles_y,
                     cudaStream_t s) {
    if (chunks == 2) {
        if (lanes == 32) return go<32, 2, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        return cudaErrorInvalidValue;
    }
    switch (lanes) {
        case 2: return go<2, 1, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        case 4: return go<4, 1, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        case 8: return go<8, 1, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        case 16: return go<16, 1, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        case 32: return go<32, 1, RED, HAS_VAL>(a, ctas_x, tiles_y, s);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace segment_detail

// Launch of the SEGMENT kernels for one reduction (instantiated per reduction
// in f_segment_{sum,max}.cu so that the variants compile in parallel).
template <int RED>
cudaError_t launch_segment_red(const RunArgs &a, int lanes, int chunks, bool has_val, int ctas_x,
                               int tiles_y, cudaStream_t s) {
    return has_val ? segment_detail::by_shape<RED, true>(a, lanes, chunks, ctas_x, tiles_y, s)
                   : segment_detail::by_shape<RED, false>(a, lanes, chunks, ctas_x, tiles_y, s);
}

extern template cudaError_t launch_segment_red<SPMM_SUM>(const RunArgs &, int, int, bool, int,
                                                         int, cudaStream_t);
extern template cudaError_t launch_segment_red<SPMM_MAX>(const RunArgs &, int, int, bool, int,
                                                         int, cudaStream_t);

}  // namespace spmm
