// WARPROW family and the heavy-row split.
//
// WARPROW: one warp per row (graph-spmm model card, "Method"). The warp is cut
// into G = 32 / L groups of L lanes; group g takes the row's entries
// g, g + G, g + 2G, ... (coalesced col/val loads across groups), lane t owns
// the column vector (blockIdx.y * L + t) * V, and the G partial accumulators
// are combined by a fixed xor-shuffle butterfly. Suited to skewed degree
// distributions: a long row keeps all 32 lanes busy even when N is narrow.
//
// Heavy-row split: rows with more than t_split entries are skipped by the
// light-row kernels. Phase 1 gives every chunk of `chunk` consecutive entries
// of such a row its own warp (same mapping as WARPROW) and writes the chunk's
// partial (sum, or (max, argmax) pair) per column to the workspace. Phase 2,
// a second launch on the same stream, combines each heavy row's chunk
// partials in chunk order and writes C. No atomics and no inter-block waits:
// the result is a pure function of the plan. (ParamSpMM section 3.2 and
// Algorithm 2: nonzero-split balancing, there combined with atomicAdd;
// DualGCN section 3.3: heavy rows get ceil(nnz/32) warps; graph-spmm model
// card, "Requirements and limits": hubs want a segmented schedule.)
#include "common.cuh"

namespace spmm {

// Reduce entries [p0, p1) of one row into `acc`; on return every group of the
// warp holds the combined result. All 32 lanes must call this.
template <int V, int L, int RED, bool HAS_VAL>
__device__ __forceinline__ void warp_segment(const RunArgs &a, int p0, int p1, int g,
                                             const float *Bv, Acc<V, RED, HAS_VAL> &acc) {
    constexpr int G = kWarp / L;
    const int64_t N = a.N;
    if constexpr (L == kWarp && RED == SPMM_MAX) {
        // Whole-warp max rows: the row's columns and values 32 at a time by one
        // coalesced load, then four gathers in flight per step, their columns
        // passed by shuffles, so only one load in 32 entries waits before its
        // gather. Same order of comparisons as below. Measured 4-10% faster
        // for max on R-MAT and Chung-Lu at N = 128 and 256; the sums were
        // 4-16% slower this way (one more live pair of registers at 32 per
        // thread) and keep the loop below.
        const int lane = threadIdx.x & (kWarp - 1);
        for (int q = p0; q < p1; q += kWarp) {
            const int n = min(kWarp, p1 - q);
            int cj = 0;
            float cw = 1.0f;
            if (lane < n) {
                cj = ld_stream(a.col + q + lane);
                if (HAS_VAL) cw = ld_stream(a.val + q + lane);
            }
            int e = 0;
            for (; e + 4 <= n; e += 4) {
                int j[4];
                float w[4], b[4][V];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    j[u] = __shfl_sync(0xffffffffu, cj, e + u);
                    w[u] = HAS_VAL ? __shfl_sync(0xffffffffu, cw, e + u) : 1.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) ld_vec<V>(Bv + (int64_t)j[u] * N, b[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc.add(w[u], j[u], b[u]);
            }
            for (; e < n; ++e) {
                const int j = __shfl_sync(0xffffffffu, cj, e);
                const float w = HAS_VAL ? __shfl_sync(0xffffffffu, cw, e) : 1.0f;
                float b[V];
                ld_vec<V>(Bv + (int64_t)j * N, b);
                acc.add(w, j, b);
            }
        }
        return;    // one group of 32 lanes: nothing to combine
    }
    int p = p0 + g;
    for (; p + 3 * G < p1; p += 4 * G) {
        int j[4];
        float w[4], b[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) j[u] = ld_stream(a.col + p + u * G);
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = HAS_VAL ? ld_stream(a.val + p + u * G) : 1.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u) ld_vec<V>(Bv + (int64_t)j[u] * N, b[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc.add(w[u], j[u], b[u]);
    }
    // The last (< 4) entries of this group. With several groups per row (L <= 16)
    // these tails are a large part of short rows: for the sum their loads are
    // issued together, predicated, so a short row costs one round trip
    // (measured 9-17% faster on the R-MAT and Chung-Lu graphs; mean, max and
    // whole-warp rows measured no faster and keep the plain loop). The order
    // of the adds is the same either way.
    if constexpr (RED == SPMM_SUM && L <= 16) {
        int j[3];
        float w[3], b[3][V];
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const bool in = p + u * G < p1;
            j[u] = in ? ld_stream(a.col + p + u * G) : 0;
            w[u] = (HAS_VAL && in) ? ld_stream(a.val + p + u * G) : 1.0f;
        }
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (p + u * G < p1) ld_vec<V>(Bv + (int64_t)j[u] * N, b[u]);
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (p + u * G < p1) acc.add(w[u], j[u], b[u]);
    } else {
        for (; p < p1; p += G) {
            const int j = ld_stream(a.col + p);
            const float w = HAS_VAL ? ld_stream(a.val + p) : 1.0f;
            float b[V];
            ld_vec<V>(Bv + (int64_t)j * N, b);
            acc.add(w, j, b);
        }
    }
#pragma unroll
    for (int off = L; off < kWarp; off <<= 1) acc.combine_xor(off);
}

// Eight CTAs per SM (32 registers a thread, a few bytes spilled in some
// instantiations): on the permuted power-law graphs the kernel waits on
// dependent DRAM loads, and 64 resident warps instead of the 48 that 40
// registers allow made the weighted sums 10-14% faster (R-MAT N=64,
// Chung-Lu N=16 and 64); max, mean and 32-lane rows were unchanged.
template <int V, int L, int RED, bool HAS_VAL>
__global__ void __launch_bounds__(256, 8) k_warprow(const RunArgs a) {
    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / L;
    const int t = lane % L;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= a.M) return;                         // uniform per warp
    const int p0 = ld_stream(a.rowptr + row);
    const int p1 = ld_stream(a.rowptr + row + 1);
    const int d = p1 - p0;
    if (d > a.t_split) return;                      // uniform per warp

    const int vi = blockIdx.y * L + t;
    const int vl = min(vi, a.n_vec - 1);
    Acc<V, RED, HAS_VAL> acc;
    acc.init();
    warp_segment<V, L, RED, HAS_VAL>(a, p0, p1, g, a.B + (int64_t)vl * V, acc);
    if (g != 0 || vi >= a.n_vec) return;
    float out[V];
    int arg[V];
    acc.finish(d, out, arg);
    const int64_t N = a.N;
    if constexpr (RED == SPMM_SUM) mean_scale<V>(a, d, out);
    epilogue<V>(a, (int64_t)vi * V, out);
    st_vec<V>(a.C + row * N + (int64_t)vi * V, out);
    if (RED == SPMM_MAX && a.argmax) st_vec_i<V>(a.argmax + row * N + (int64_t)vi * V, arg);
}

// Phase 1: one warp per heavy-row chunk; raw partials to the workspace.
template <int V, int L, int RED, bool HAS_VAL>
__global__ void __launch_bounds__(256) k_heavy_chunks(const RunArgs a) {
    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / L;
    const int t = lane % L;
    const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (c >= a.n_chunks) return;                    // uniform per warp
    const int2 rc = a.chunks[c];                    // (row, first entry)
    const int row_end = ld_stream(a.rowptr + rc.x + 1);
    const int p0 = rc.y;
    const int p1 = min(p0 + a.chunk, row_end);

    const int vi = blockIdx.y * L + t;
    const int vl = min(vi, a.n_vec - 1);
    Acc<V, RED, HAS_VAL> acc;
    acc.init();
    warp_segment<V, L, RED, HAS_VAL>(a, p0, p1, g, a.B + (int64_t)vl * V, acc);
    if (g != 0 || vi >= a.n_vec) return;
    const int64_t o = c * (int64_t)a.N + (int64_t)vi * V;
    float v[V];
#pragma unroll
    for (int e = 0; e < V; ++e) v[e] = acc.v[e];
    st_vec<V>(a.ws_val + o, v);
    if constexpr (RED == SPMM_MAX) st_vec_i<V>(a.ws_arg + o, acc.j);
}

// Phase 2: one block per heavy row; each thread combines the row's chunk
// partials for its column vectors in chunk order.
template <int V, int RED>
__global__ void __launch_bounds__(128) k_heavy_combine(const RunArgs a) {
    const int h = blockIdx.x;
    const int row = a.heavy_rows[h];
    const int c0 = a.heavy_chunk0[h];
    const int c1 = a.heavy_chunk0[h + 1];
    const int d = a.rowptr[row + 1] - a.rowptr[row];
    const int64_t N = a.N;
    for (int vi = blockIdx.y * blockDim.x + threadIdx.x; vi < a.n_vec;
         vi += gridDim.y * blockDim.x) {
        float acc[V];
        int arg[V];
        const int64_t col0 = (int64_t)vi * V;
        ld_vec<V>(a.ws_val + c0 * N + col0, acc);
        if constexpr (RED == SPMM_MAX) {
            if constexpr (V == 4) {
                const int4 q = __ldg(reinterpret_cast<const int4 *>(a.ws_arg + c0 * N + col0));
                arg[0] = q.x; arg[1] = q.y; arg[2] = q.z; arg[3] = q.w;
            } else {
                arg[0] = __ldg(a.ws_arg + c0 * N + col0);
            }
        }
        for (int c = c0 + 1; c < c1; ++c) {
            float x[V];
            ld_vec<V>(a.ws_val + c * N + col0, x);
            if constexpr (RED == SPMM_MAX) {
                int xj[V];
                if constexpr (V == 4) {
                    const int4 q = __ldg(reinterpret_cast<const int4 *>(a.ws_arg + c * N + col0));
                    xj[0] = q.x; xj[1] = q.y; xj[2] = q.z; xj[3] = q.w;
                } else {
                    xj[0] = __ldg(a.ws_arg + c * N + col0);
                }
#pragma unroll
                for (int e = 0; e < V; ++e)
                    if (max_better(x[e], xj[e], acc[e], arg[e])) { acc[e] = x[e]; arg[e] = xj[e]; }
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
            }
        }
        if constexpr (RED == SPMM_MEAN) {
            const float inv_d = rcp_approx((float)d);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = __fmul_rn(acc[e], inv_d);
        }
        if constexpr (RED == SPMM_SUM) mean_scale<V>(a, d, acc);
        epilogue<V>(a, col0, acc);
        st_vec<V>(a.C + (int64_t)row * N + col0, acc);
        if constexpr (RED == SPMM_MAX) {
            if (a.argmax) st_vec_i<V>(a.argmax + (int64_t)row * N + col0, arg);
        }
    }
}

namespace {
constexpr int kThreads = 256;

template <int V, int L, int RED, bool HAS_VAL>
cudaError_t go_rows(const RunArgs &a, int tiles, cudaStream_t s) {
    const int64_t warps_per_block = kThreads / kWarp;
    const int64_t blocks = (a.M + warps_per_block - 1) / warps_per_block;
    k_warprow<V, L, RED, HAS_VAL><<<dim3((unsigned)blocks, (unsigned)tiles), kThreads, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int V, int L, int RED, bool HAS_VAL>
cudaError_t go_heavy(const RunArgs &a, int tiles, cudaStream_t s) {
    const int64_t warps_per_block = kThreads / kWarp;
    const int64_t blocks = (a.n_chunks + warps_per_block - 1) / warps_per_block;
    k_heavy_chunks<V, L, RED, HAS_VAL>
        <<<dim3((unsigned)blocks, (unsigned)tiles), kThreads, 0, s>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int ty = (int)std::min<int64_t>((a.n_vec + 127) / 128, 64);
    k_heavy_combine<V, RED><<<dim3((unsigned)a.n_heavy, (unsigned)ty), 128, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int V, int RED, bool HAS_VAL, bool HEAVY>
cudaError_t by_lanes(const RunArgs &a, int lanes, int tiles, cudaStream_t s) {
#define SPMM_CASE(LL)                                                        \
    case LL:                                                                 \
        return HEAVY ? go_heavy<V, LL, RED, HAS_VAL>(a, tiles, s)            \
                     : go_rows<V, LL, RED, HAS_VAL>(a, tiles, s);
    switch (lanes) {
        SPMM_CASE(2)
        SPMM_CASE(4)
        SPMM_CASE(8)
        SPMM_CASE(16)
        SPMM_CASE(32)
        default: return cudaErrorInvalidValue;
    }
#undef SPMM_CASE
}

template <bool HEAVY>
cudaError_t dispatch(const RunArgs &a_in, int vec, int lanes, int reduce, bool has_val, int tiles,
                     cudaStream_t s) {
    // The mean runs as the sum kernel with a final 1/d (mean_scale: the same
    // arithmetic as a MEAN instantiation's finish, so the same bits). The sum
    // kernel's batched tail and its register budget make it faster: 18% on the
    // 4M-row Chung-Lu graph at N=128 and 256, 7-8% at N=16 and 64.
    RunArgs a = a_in;
    if (reduce == SPMM_MEAN) {
        a.mean = 1;
        reduce = SPMM_SUM;
    }
#define SPMM_RED(V, R)                                                                  \
    return has_val ? by_lanes<V, R, true, HEAVY>(a, lanes, tiles, s)                    \
                   : by_lanes<V, R, false, HEAVY>(a, lanes, tiles, s);
    if (vec == 4) {
        switch (reduce) {
            case SPMM_SUM: SPMM_RED(4, SPMM_SUM)
            case SPMM_MAX: SPMM_RED(4, SPMM_MAX)
        }
    } else {
        switch (reduce) {
            case SPMM_SUM: SPMM_RED(1, SPMM_SUM)
            case SPMM_MAX: SPMM_RED(1, SPMM_MAX)
        }
    }
#undef SPMM_RED
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_warprow(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                           int tiles, cudaStream_t s) {
    return dispatch<false>(a, vec, lanes, reduce, has_val, tiles, s);
}

cudaError_t launch_heavy(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                         int tiles, cudaStream_t s) {
    return dispatch<true>(a, vec, lanes, reduce, has_val, tiles, s);
}

}  // namespace spmm
