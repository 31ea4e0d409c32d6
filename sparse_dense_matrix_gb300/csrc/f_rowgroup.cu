// ROWGROUP family: several rows per warp, for graphs whose row degrees are
// nearly uniform (low degree CV).
//
// A warp is cut into G = 32 / L groups of L lanes; group g owns one row and
// walks all of the row's entries in CSR order. Lane t of the group owns the
// vector of `V` feature columns (blockIdx.y * L + t) * V, so the gathered B row
// slice is one coalesced 16*L-byte (V = 4) read per entry and every output
// element reduces privately in a register (no shuffles, no atomics). Four
// entries are in flight per lane (independent loads before the FMAs).
//
// This is the narrow-N mapping of the graph-spmm model card ("Method": one
// warp per row, lanes hold strided slices of the feature columns), folded so
// that N / 4 < 32 does not leave lanes idle (ParamSpMM section 3.3, Eq. (1):
// the MAC-job gap when N is not a multiple of the lanes' columns).
#include "common.cuh"

namespace spmm {

template <int V, int L, int RED, bool HAS_VAL>
__global__ void __launch_bounds__(256) k_rowgroup(const RunArgs a) {
    constexpr int G = kWarp / L;
    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / L;
    const int t = lane % L;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t row = warp * G + g;
    if (row >= a.M) return;
    const int p0 = ld_stream(a.rowptr + row);
    const int p1 = ld_stream(a.rowptr + row + 1);
    const int d = p1 - p0;
    if (d > a.t_split) return;                      // written by the heavy-row split

    const int vi = blockIdx.y * L + t;              // this lane's column vector
    const int vl = min(vi, a.n_vec - 1);            // clamped for loads of idle lanes
    const float *Bv = a.B + (int64_t)vl * V;
    const int64_t N = a.N;

    Acc<V, RED, HAS_VAL> acc;
    acc.init();
    int p = p0;
    for (; p + 4 <= p1; p += 4) {
        int j[4];
        float w[4], b[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) j[u] = ld_stream(a.col + p + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = HAS_VAL ? ld_stream(a.val + p + u) : 1.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u) ld_vec<V>(Bv + (int64_t)j[u] * N, b[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc.add(w[u], j[u], b[u]);
    }
    // the last (< 4) entries: for the sum with narrow rows of lanes their
    // loads are issued together, predicated (one round trip); the order of
    // the adds is the same either way
    if constexpr (RED == SPMM_SUM && L <= 16) {
        int j[3];
        float w[3], b[3][V];
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const bool in = p + u < p1;
            j[u] = in ? ld_stream(a.col + p + u) : 0;
            w[u] = (HAS_VAL && in) ? ld_stream(a.val + p + u) : 1.0f;
        }
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (p + u < p1) ld_vec<V>(Bv + (int64_t)j[u] * N, b[u]);
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (p + u < p1) acc.add(w[u], j[u], b[u]);
    } else {
        for (; p < p1; ++p) {
            const int j = ld_stream(a.col + p);
            const float w = HAS_VAL ? ld_stream(a.val + p) : 1.0f;
            float b[V];
            ld_vec<V>(Bv + (int64_t)j * N, b);
            acc.add(w, j, b);
        }
    }
    if (vi >= a.n_vec) return;
    float out[V];
    int arg[V];
    acc.finish(d, out, arg);
    if constexpr (RED == SPMM_SUM) mean_scale<V>(a, d, out);
    epilogue<V>(a, (int64_t)vi * V, out);
    st_vec<V>(a.C + row * N + (int64_t)vi * V, out);
    if (RED == SPMM_MAX && a.argmax) st_vec_i<V>(a.argmax + row * N + (int64_t)vi * V, arg);
}

namespace {
template <int V, int L, int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, int tiles, cudaStream_t s) {
    constexpr int kThreads = 256;
    constexpr int rows_per_block = (kThreads / kWarp) * (kWarp / L);
    const int64_t blocks = (a.M + rows_per_block - 1) / rows_per_block;
    dim3 grid((unsigned)blocks, (unsigned)tiles);
    k_rowgroup<V, L, RED, HAS_VAL><<<grid, kThreads, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int V, int RED, bool HAS_VAL>
cudaError_t by_lanes(const RunArgs &a, int lanes, int tiles, cudaStream_t s) {
    switch (lanes) {
        case 2: return go<V, 2, RED, HAS_VAL>(a, tiles, s);
        case 4: return go<V, 4, RED, HAS_VAL>(a, tiles, s);
        case 8: return go<V, 8, RED, HAS_VAL>(a, tiles, s);
        case 16: return go<V, 16, RED, HAS_VAL>(a, tiles, s);
        case 32: return go<V, 32, RED, HAS_VAL>(a, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int V, int RED>
cudaError_t by_val(const RunArgs &a, bool has_val, int lanes, int tiles, cudaStream_t s) {
    return has_val ? by_lanes<V, RED, true>(a, lanes, tiles, s)
                   : by_lanes<V, RED, false>(a, lanes, tiles, s);
}

template <int V>
cudaError_t by_reduce(const RunArgs &a, int reduce, bool has_val, int lanes, int tiles,
                      cudaStream_t s) {
    switch (reduce) {
        case SPMM_SUM: return by_val<V, SPMM_SUM>(a, has_val, lanes, tiles, s);
        case SPMM_MEAN:
            if (lanes == 32) {
                // whole-warp rows: the mean as the sum with a final 1/d (as in WARPROW)
                RunArgs m = a;
                m.mean = 1;
                return by_val<V, SPMM_SUM>(m, has_val, lanes, tiles, s);
            }
            return by_val<V, SPMM_MEAN>(a, has_val, lanes, tiles, s);
        case SPMM_MAX: return by_val<V, SPMM_MAX>(a, has_val, lanes, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_rowgroup(const RunArgs &a, int vec, int lanes, int reduce, bool has_val,
                            int tiles, cudaStream_t s) {
    return vec == 4 ? by_reduce<4>(a, reduce, has_val, lanes, tiles, s)
                    : by_reduce<1>(a, reduce, has_val, lanes, tiles, s);
}

}  // namespace spmm
