// STREAM family: the stored entries as one stream, cut into equal contiguous
// ranges, each walked by one lane group of L lanes (ParamSpMM section 3.2,
// nonzero-split workload balancing; DualGCN section 3.3: independent gathers
// in flight).
//
// A row-per-warp kernel pays each row's dependent chain (row pointers, then
// columns, then the B rows) once per row, and a short row leaves most of a
// batch of gathers empty. Here a lane group walks the entries of its range
// in CSR order with the plan's per-entry row ids: the columns, values and row
// ids of the next 32 entries are loaded while the current 32 are gathered, U
// B rows at a time, so the gathers of consecutive rows overlap and nothing
// waits on a row pointer. A row is finished (mean, epilogue, store) when the
// next entry's row id differs, and the rows with no entry in between are
// written as empty rows. The groups of a warp walk different ranges and
// never exchange data. The rows open at the two ends of a range leave as
// partials that k_segment_fix combines in range order, as for the SEGMENT
// family: every summation order is fixed by the plan, N and the grid
// (bitwise reproducible, no atomics).
#pragma once

#include "common.cuh"
#include "segment.cuh"

namespace spmm {

constexpr int kStBatch = 32;    // entries whose metadata a lane group holds per batch
#ifndef SPMM_ST_U
#define SPMM_ST_U 4
#endif
#ifndef SPMM_ST_MINB
#define SPMM_ST_MINB 4
#endif
constexpr int kStU = SPMM_ST_U;          // B rows in flight per lane
constexpr int kStMinBlocks = SPMM_ST_MINB;
constexpr int kStThreads = 256;

// Entry e of a batch is held by lane e % L of its group, in register e / L.
template <int PER, int L, typename T>
__device__ __forceinline__ T st_pick(const T (&x)[PER], int e) {
    T y = x[0];
#pragma unroll
    for (int k = 1; k < PER; ++k)
        if (e / L == k) y = x[k];
    return y;
}

// L lanes per range, each owning one float4 of the range's 4L-column tile.
template <int L, int RED, bool HAS_VAL, bool EPI>
__global__ void __launch_bounds__(kStThreads, kStMinBlocks) k_stream(const RunArgs a) {
    constexpr int G = kWarp / L;            // ranges per warp
    constexpr int PER = kStBatch / L;       // entries of a batch held per lane
    constexpr int U = kStU;
    static_assert(kStBatch % U == 0 && kStBatch % L == 0, "batch shape");
    using A = Acc<4, RED, HAS_VAL>;
    const int lane = threadIdx.x & (kWarp - 1), g = lane / L, t = lane % L;
    const unsigned gmask = L == kWarp ? 0xffffffffu : ((1u << L) - 1u) << (g * L);
    const int64_t R = a.seg_warps;          // ranges of the grid
    const int64_t v = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * G + g;
    if (v >= R) return;                     // uniform per group
    const int64_t nnz = a.rowptr[a.M];
    // the host makes R <= nnz, so no range is empty
    const int64_t e0 = nnz * v / R, e1 = nnz * (v + 1) / R;
    const int64_t N = a.N;
    constexpr int CW = 4 * L;               // columns of the tile
    const int64_t c = (int64_t)blockIdx.y * CW + 4 * t;
    const bool act = c < N;
    const float *Bl = a.B + (act ? c : N - 4);

    auto store_row = [&](int64_t row, const A &x, int d) {
        if (!act) return;
        float out[4];
        int arg[4];
        x.finish(d, out, arg);
        if constexpr (RED == SPMM_SUM) mean_scale<4>(a, d, out);
        if constexpr (EPI) epilogue<4>(a, c, out);
        st_vec<4>(a.C + row * N + c, out);
        if (RED == SPMM_MAX && a.argmax) st_vec_i<4>(a.argmax + row * N + c, arg);
    };
    auto empty_rows = [&](int64_t r0, int64_t r1) {   // rows [r0, r1) hold no entry
        A z;
        z.init();
        for (int64_t r = r0; r < r1; ++r) store_row(r, z, 0);
    };
    // slot 0: the row open at the start of the range, slot 1: at its end
    auto store_carry = [&](int slot, const A &x) {
        if (!act) return;
        const int64_t o = (((int64_t)blockIdx.y * R + v) * 2 + slot) * CW + 4 * t;
        float w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = x.v[e];
        st_vec<4>(a.seg_cval + o, w);
        if constexpr (RED == SPMM_MAX) st_vec_i<4>(a.seg_carg + o, x.j);
    };

    // entry base + k L + t for k < PER (lane t of the group holds entries t, L + t, ...)
    int mc[PER], mr[PER], nc[PER], nr[PER];
    float mv[PER], nv[PER];
    auto load_batch = [&](int64_t base, int (&cc)[PER], int (&rr)[PER], float (&ww)[PER]) {
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int64_t p = base + k * L + t;
            const bool in = p < e1;
            cc[k] = in ? ld_stream(a.col + p) : 0;
            rr[k] = in ? ld_stream(a.ga_rid + p) : -1;
            ww[k] = (HAS_VAL && in) ? ld_stream(a.val + p) : 1.0f;
        }
    };

    const int first_row = a.ga_rid[e0], last_row = a.ga_rid[e1 - 1];
    const bool head_open = e0 > 0 && a.ga_rid[e0 - 1] == first_row;
    const bool tail_open = e1 < nnz && a.ga_rid[e1] == last_row;
    const int64_t next_row = e1 < nnz ? (int64_t)a.ga_rid[e1] : a.M;
    if (e0 == 0) empty_rows(0, first_row);

    A acc;
    acc.init();
    int cur = first_row, cnt = 0, h0_ends = 0, tail_row = -1;
    bool head = head_open;
    load_batch(e0, mc, mr, mv);
    for (int64_t b = e0; b < e1; b += kStBatch) {
        if (b + kStBatch < e1) load_batch(b + kStBatch, nc, nr, nv);
        const int n = (int)(e1 - b < kStBatch ? e1 - b : kStBatch);
#pragma unroll 1
        for (int s0 = 0; s0 < n; s0 += U) {
            int j[U];
            float bv[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = s0 + u;
                j[u] = __shfl_sync(gmask, st_pick<PER, L>(mc, e), e % L, L);
                if (e < n) ld_vec<4>(Bl + (int64_t)j[u] * N, bv[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = s0 + u;
                const int r = __shfl_sync(gmask, st_pick<PER, L>(mr, e), e % L, L);
                const float w =
                    HAS_VAL ? __shfl_sync(gmask, st_pick<PER, L>(mv, e), e % L, L) : 1.0f;
                if (e < n) {
                    if (r != cur) {                 // row `cur` ended at the previous entry
                        if (head) {
                            store_carry(0, acc);
                            h0_ends = 1;
                            head = false;
                        } else {
                            store_row(cur, acc, cnt);
                        }
                        empty_rows((int64_t)cur + 1, r);
                        cur = r;
                        cnt = 0;
                        acc.init();
                    }
                    acc.add(w, j[u], bv[u]);
                    ++cnt;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            mc[k] = nc[k];
            mr[k] = nr[k];
            mv[k] = nv[k];
        }
    }
    if (tail_open) {                                // the last row goes on past e1
        if (head) {
            store_carry(0, acc);
            h0_ends = 0;
        } else {
            store_carry(1, acc);
            tail_row = cur;
        }
    } else {
        if (head) {
            store_carry(0, acc);
            h0_ends = 1;
        } else {
            store_row(cur, acc, cnt);
        }
        empty_rows((int64_t)cur + 1, next_row);
    }
    if (t == 0 && blockIdx.y == 0)
        a.seg_meta[v] = make_int4(head_open ? first_row : -1, h0_ends, tail_row, 0);
}

namespace stream_detail {
template <int L, int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, int64_t warps, int tiles_y, cudaStream_t s) {
    const bool epi = a.bias != nullptr || a.act != SPMM_ACT_NONE;
    auto kern = epi ? k_stream<L, RED, HAS_VAL, true> : k_stream<L, RED, HAS_VAL, false>;
    const int64_t blocks = (warps + kStThreads / kWarp - 1) / (kStThreads / kWarp);
    kern<<<dim3((unsigned)blocks, (unsigned)tiles_y), kStThreads, 0, s>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = (int64_t)a.seg_warps * (a.N / 4);
    k_segment_fix<RED><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a, 4 * L);
    count_launch();
    return cudaGetLastError();
}
}  // namespace stream_detail

// Launch for one reduction (instantiated per reduction in f_stream_{sum,max}.cu).
// a.seg_warps holds the number of ranges, a.seg_meta / seg_cval / seg_carg
// the open-row workspace.
template <int RED>
cudaError_t launch_stream_red(const RunArgs &a, int lanes, bool has_val, int tiles_y,
                              cudaStream_t s) {
    const int64_t groups = kWarp / lanes;
    const int64_t warps = (a.seg_warps + groups - 1) / groups;
    if (lanes == 32)
        return has_val ? stream_detail::go<32, RED, true>(a, warps, tiles_y, s)
                       : stream_detail::go<32, RED, false>(a, warps, tiles_y, s);
    if (lanes == 16)
        return has_val ? stream_detail::go<16, RED, true>(a, warps, tiles_y, s)
                       : stream_detail::go<16, RED, false>(a, warps, tiles_y, s);
    return cudaErrorInvalidValue;
}

extern template cudaError_t launch_stream_red<SPMM_SUM>(const RunArgs &, int, bool, int,
                                                        cudaStream_t);
extern template cudaError_t launch_stream_red<SPMM_MAX>(const RunArgs &, int, bool, int,
                                                        cudaStream_t);

}  // namespace spmm
