// Backward support (graph-spmm card, "Requirements and limits": the backward
// of a sum aggregation is the transposed product, composed from a second
// adjacency on the reversed edge list; "API": the argmax of spmm_max feeds the
// max-pool backward).
//
// spmm_transpose builds A^T in CSR on the device: a stable LSD radix sort of
// the entries by column (8-bit digits, tiles of 4096 entries; within a tile
// the rank of an entry among equal digits comes from warp matching and
// per-warp digit counts, so placement is a pure function of the input - no
// atomics), then a gather of rows and values and the new row pointers. Stable
// on CSR order means the entries of a column come out in increasing row.
// spmm_maxpool_backward reduces, for every column j of A, dC[i, k] * a_ij over
// the entries (i, j) whose row chose j as argmax[i, k], one stored copy (the
// one whose product won) per duplicated pair.
#include <vector>

#include "common.cuh"

namespace spmm {
namespace {

// ------------------------------------------------------------- block scan
constexpr int kScanThreads = 1024;

// exclusive scan of one value per thread over a 1024-thread block
__device__ __forceinline__ int warp_inclusive_scan(int x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
    }
    return x;
}

__device__ __forceinline__ int block_exclusive_scan(int x, int *total) {
    __shared__ int warp_excl[32];
    __shared__ int s_total;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int incl = warp_inclusive_scan(x, lane);
    if (lane == 31) warp_excl[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int s = warp_excl[lane];
        const int si = warp_inclusive_scan(s, lane);
        warp_excl[lane] = si - s;
        if (lane == 31) s_total = si;
    }
    __syncthreads();
    const int excl = incl - x + warp_excl[w];
    *total = s_total;
    __syncthreads();   // the shared words are reused by the next call
    return excl;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_local(const int *in, int *out, int64_t n,
                                                            int *bsum) {
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    const int x = i < n ? in[i] : 0;
    int total;
    const int e = block_exclusive_scan(x, &total);
    if (i < n) out[i] = e;
    if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_bsums(int *bsum, int64_t nb) {
    int carry = 0;
    for (int64_t base = 0; base < nb; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        const int x = i < nb ? bsum[i] : 0;
        int total;
        const int e = block_exclusive_scan(x, &total);
        if (i < nb) bsum[i] = e + carry;
        carry += total;
    }
}

__global__ void k_scan_add(int *out, int64_t n, const int *bsum) {
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    if (i < n) out[i] += bsum[blockIdx.x];
}

// ------------------------------------------------------------- radix sort
constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
constexpr int kRIters = 16;
constexpr int kRTile = kRThreads * kRIters;   // entries per tile
constexpr int kRBins = 256;

__global__ void __launch_bounds__(kRThreads) k_radix_hist(const uint32_t *keys, int64_t n,
                                                         int shift, int64_t T, int *hist) {
    __shared__ int cnt[kRBins];
    cnt[threadIdx.x] = 0;
    __syncthreads();
    for (int it = 0; it < kRIters; ++it) {
        const int64_t idx = (int64_t)blockIdx.x * kRTile + it * kRThreads + threadIdx.x;
        if (idx < n) atomicAdd(&cnt[(keys[idx] >> shift) & 255u], 1);
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * T + blockIdx.x] = cnt[threadIdx.x];
}

// Stable scatter: entry idx of tile b, digit d, goes to
// offs[d][b] + (earlier entries of the tile with digit d).
__global__ void __launch_bounds__(kRThreads) k_radix_scatter(const uint32_t *kin,
                                                            const int32_t *vin, uint32_t *kout,
                                                            int32_t *vout, int64_t n, int shift,
                                                            int64_t T, const int *offs) {
    __shared__ int counter[kRBins];
    __shared__ int wcnt[kRWarps][kRBins + 1];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    counter[threadIdx.x] = 0;
    __syncthreads();
    for (int it = 0; it < kRIters; ++it) {
        const int64_t idx = (int64_t)blockIdx.x * kRTile + it * kRThreads + threadIdx.x;
        const bool valid = idx < n;
        const uint32_t key = valid ? kin[idx] : 0u;
        const int d = valid ? (int)((key >> shift) & 255u) : kRBins;   // kRBins: no entry
        const int32_t v = valid ? (vin ? vin[idx] : (int32_t)idx) : 0;
#pragma unroll
        for (int q = 0; q < kRWarps; ++q) wcnt[q][threadIdx.x] = 0;
        if (threadIdx.x == 0)
            for (int q = 0; q < kRWarps; ++q) wcnt[q][kRBins] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (rank == 0) wcnt[w][d] = __popc(peers);
        __syncthreads();
        if (valid) {
            int before = 0;
            for (int q = 0; q < w; ++q) before += wcnt[q][d];
            const int64_t pos = (int64_t)offs[(int64_t)d * T + blockIdx.x] + counter[d] + before + rank;
            kout[pos] = key;
            vout[pos] = v;
        }
        __syncthreads();
        int add = 0;
#pragma unroll
        for (int q = 0; q < kRWarps; ++q) add += wcnt[q][threadIdx.x];
        counter[threadIdx.x] += add;
        __syncthreads();
    }
}

// ------------------------------------------------------- transpose kernels
__global__ void k_row_of(const int32_t *rowptr, int64_t M, int32_t *row_of) {
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < M; i += warps)
        for (int p = rowptr[i] + lane; p < rowptr[i + 1]; p += 32) row_of[p] = (int32_t)i;
}

__global__ void k_gather_t(const int32_t *perm, const int32_t *row_of, const int32_t *rowptr,
                           const float *val, int64_t nnz, int scale_mean, int32_t *colT,
                           float *valT) {
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nnz;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int p = perm[q];
        const int i = row_of[p];
        colT[q] = i;
        if (valT) {
            const float a = val ? val[p] : 1.0f;
            // a / d_i in fp64, rounded once to fp32 (d_i is exact in fp64)
            valT[q] = scale_mean
                          ? __double2float_rn(__ddiv_rn((double)a, (double)(rowptr[i + 1] - rowptr[i])))
                          : a;
        }
    }
}

// rowptrT[j] = number of sorted keys below j (a lower bound by binary search)
__global__ void k_bounds(const uint32_t *keys, int64_t nnz, int64_t K, int32_t *rowptrT) {
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j <= K;
         j += (int64_t)gridDim.x * blockDim.x) {
        int64_t lo = 0, hi = nnz;
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if ((int64_t)keys[mid] < j) lo = mid + 1; else hi = mid;
        }
        rowptrT[j] = (int32_t)lo;
    }
}

// ------------------------------------------------------ max-pool backward
// Row j of A^T lists the entries (i, a_ij) of column j of A in increasing i;
// copies of a duplicated pair (i, j) are adjacent, in their CSR order. The
// forward maximum of row i took its value from one stored entry, so for each
// run of copies of one i only the copy with the largest fp32 product
// a * B[j, c] (the first on equal products) passes the gradient:
// dB[j, c] = sum over the runs with argmax[i, c] == j of a_w * dC[i, c],
// accumulated in fp32 in increasing i (graph-spmm card, "Correctness":
// duplicated pairs are legal CSR; "API": the argmax feeds this backward).
// L lanes own a row, V columns per lane per step; a warp holds 32 / L rows.
// Rows of A^T longer than t_split (hub columns of A) are left to the split
// below, as in the forward product.
//
// mp_accumulate covers entries [p0, p1) of row j, which spans [r0, r1). A run
// that began before p0 belongs to the previous chunk and is skipped; a run
// that reaches p1 is followed to its end. bj: B[j, c .. c + V) (weighted A).
template <int V, bool HAS_VAL>
__device__ __forceinline__ void mp_accumulate(const int32_t *__restrict__ colT,
                                              const float *__restrict__ valT,
                                              const int32_t *__restrict__ argmax,
                                              const float *__restrict__ dC, int64_t N, int j,
                                              int r0, int p0, int p1, int r1, int64_t c,
                                              const float (&bj)[V], float (&acc)[V]) {
    int p = p0;
    if (p > r0 && p < p1) {
        const int prev = colT[p - 1];
        while (p < p1 && colT[p] == prev) ++p;
    }
    while (p < p1) {
        const int64_t i = colT[p];
        float aw[V];
        {
            const float a = HAS_VAL ? valT[p] : 1.0f;
#pragma unroll
            for (int e = 0; e < V; ++e) aw[e] = a;
        }
        int q = p + 1;
        if constexpr (HAS_VAL) {
            float yw[V];
#pragma unroll
            for (int e = 0; e < V; ++e) yw[e] = __fmul_rn(aw[e], bj[e]);
            for (; q < r1 && colT[q] == (int)i; ++q) {
                const float a = valT[q];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float y = __fmul_rn(a, bj[e]);
                    if (y > yw[e]) { yw[e] = y; aw[e] = a; }
                }
            }
        } else {
            while (q < r1 && colT[q] == (int)i) ++q;
        }
        float g[V];
        int w[V];
        if constexpr (V == 4) {
            const float4 gv = __ldg(reinterpret_cast<const float4 *>(dC + i * N + c));
            const int4 wv = __ldg(reinterpret_cast<const int4 *>(argmax + i * N + c));
            g[0] = gv.x; g[1] = gv.y; g[2] = gv.z; g[3] = gv.w;
            w[0] = wv.x; w[1] = wv.y; w[2] = wv.z; w[3] = wv.w;
        } else {
            g[0] = __ldg(dC + i * N + c);
            w[0] = __ldg(argmax + i * N + c);
        }
#pragma unroll
        for (int e = 0; e < V; ++e)
            if (w[e] == j) acc[e] = HAS_VAL ? __fmaf_rn(aw[e], g[e], acc[e]) : __fadd_rn(acc[e], g[e]);
        p = q;
    }
}

template <int V, bool HAS_VAL>
__device__ __forceinline__ void mp_brow(const float *__restrict__ B, int64_t N, int64_t j,
                                        int64_t c, float (&bj)[V]) {
#pragma unroll
    for (int e = 0; e < V; ++e) bj[e] = 0.0f;
    if constexpr (HAS_VAL) ld_vec<V>(B + j * N + c, bj);
}

template <int V, bool HAS_VAL>
__global__ void __launch_bounds__(256) k_maxpool_bwd(const int32_t *__restrict__ rowptrT,
                                                    const int32_t *__restrict__ colT,
                                                    const float *__restrict__ valT,
                                                    const float *__restrict__ B,
                                                    const int32_t *__restrict__ argmax,
                                                    const float *__restrict__ dC, int64_t rows,
                                                    int64_t N, int lanes, int t_split,
                                                    float *__restrict__ dB) {
    const int lane = threadIdx.x & 31;
    const int sub = lane % lanes, grp = lane / lanes, groups = 32 / lanes;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t j = warp * groups + grp;
    if (j >= rows) return;
    const int p0 = rowptrT[j], p1 = rowptrT[j + 1];
    if (p1 - p0 > t_split) return;                 // a split row
    for (int64_t c = (int64_t)sub * V; c < N; c += (int64_t)lanes * V) {
        float acc[V], bj[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.0f;
        mp_brow<V, HAS_VAL>(B, N, j, c, bj);
        mp_accumulate<V, HAS_VAL>(colT, valT, argmax, dC, N, (int)j, p0, p0, p1, p1, c, bj, acc);
        st_vec<V>(dB + j * N + c, acc);
    }
}

// Split rows, phase 1: a warp per chunk of `chunk` entries writes its partial
// (chunk-local masked sum) to ws[q][:].
template <int V, bool HAS_VAL>
__global__ void __launch_bounds__(256) k_maxpool_chunks(const int32_t *__restrict__ rowptrT,
                                                       const int32_t *__restrict__ colT,
                                                       const float *__restrict__ valT,
                                                       const float *__restrict__ B,
                                                       const int32_t *__restrict__ argmax,
                                                       const float *__restrict__ dC, int64_t N,
                                                       const int2 *__restrict__ chunks,
                                                       int64_t n_chunks, int chunk,
                                                       float *__restrict__ ws) {
    const int lane = threadIdx.x & 31;
    const int64_t q = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (q >= n_chunks) return;
    const int2 ch = chunks[q];                      // (row of A^T, first entry)
    const int r0 = rowptrT[ch.x], r1 = rowptrT[ch.x + 1];
    const int p1 = min(ch.y + chunk, r1);
    for (int64_t c = (int64_t)lane * V; c < N; c += 32 * V) {
        float acc[V], bj[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.0f;
        mp_brow<V, HAS_VAL>(B, N, ch.x, c, bj);
        mp_accumulate<V, HAS_VAL>(colT, valT, argmax, dC, N, ch.x, r0, ch.y, p1, r1, c, bj, acc);
        st_vec<V>(ws + q * N + c, acc);
    }
}

// Split rows, phase 2: a warp per split row adds its chunks' partials in
// chunk order and writes the row of dB.
template <int V>
__global__ void __launch_bounds__(256) k_maxpool_combine(const int32_t *__restrict__ heavy_rows,
                                                        const int32_t *__restrict__ heavy_chunk0,
                                                        int64_t n_heavy, int64_t N,
                                                        const float *__restrict__ ws,
                                                        float *__restrict__ dB) {
    const int lane = threadIdx.x & 31;
    const int64_t h = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (h >= n_heavy) return;
    const int64_t j = heavy_rows[h];
    const int q0 = heavy_chunk0[h], q1 = heavy_chunk0[h + 1];
    for (int64_t c = (int64_t)lane * V; c < N; c += 32 * V) {
        float acc[V];
        ld_vec<V>(ws + (int64_t)q0 * N + c, acc);
        for (int q = q0 + 1; q < q1; ++q) {
            float x[V];
            ld_vec<V>(ws + (int64_t)q * N + c, x);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
        }
        st_vec<V>(dB + j * N + c, acc);
    }
}

// ------------------------------------------------------------------ host
cudaError_t t_alloc(void **p, size_t bytes) {
    *p = nullptr;
    return cudaMalloc(p, bytes ? bytes : 16);
}

spmm_status t_status(cudaError_t e) {
    if (e == cudaSuccess) return SPMM_OK;
    if (e == cudaErrorMemoryAllocation) return SPMM_ERR_OOM;
    return SPMM_ERR_CUDA;
}

int64_t grid_for(int64_t work, int threads, int num_sms) {
    const int64_t b = (work + threads - 1) / threads;
    return std::max<int64_t>(1, std::min<int64_t>(b, (int64_t)num_sms * 16));
}

// exclusive scan of n ints on the device (in -> out; bsum: ceil(n / 1024) ints)
cudaError_t device_scan(const int *in, int *out, int64_t n, int *bsum, cudaStream_t s) {
    const int64_t nb = (n + kScanThreads - 1) / kScanThreads;
    if (nb == 0) return cudaSuccess;
    k_scan_local<<<(unsigned)nb, kScanThreads, 0, s>>>(in, out, n, bsum);
    k_scan_bsums<<<1, kScanThreads, 0, s>>>(bsum, nb);
    k_scan_add<<<(unsigned)nb, kScanThreads, 0, s>>>(out, n, bsum);
    count_launch(3);
    return cudaGetLastError();
}

}  // namespace
}  // namespace spmm

extern "C" {

spmm_status spmm_transpose(spmm_plan_t plan, const int32_t *col, const float *val, int scale_mean,
                           int32_t *rowptrT, int32_t *colT, float *valT, void *stream) {
    using namespace spmm;
    if (!plan || !rowptrT) return SPMM_ERR_INVALID_ARG;
    const Plan *p = reinterpret_cast<const Plan *>(plan);
    const int64_t nnz = p->nnz, K = p->K;
    if (nnz > 0 && (!col || !colT)) return SPMM_ERR_INVALID_ARG;
    if (nnz > 0 && !valT && (val || scale_mean)) return SPMM_ERR_INVALID_ARG;
    // a row-range plan reads its rows' entries out of the full arrays
    col += p->col_base;
    if (val) val += p->col_base;
    cudaStream_t s = (cudaStream_t)stream;
    const int sms = p->num_sms > 0 ? p->num_sms : 1;

    cudaError_t e = cudaSuccess;
    if (nnz == 0) {
        e = cudaMemsetAsync(rowptrT, 0, sizeof(int32_t) * (size_t)(K + 1), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        return t_status(e);
    }
    // keys lie in [0, K): 8-bit digits over ceil(log2 K) bits, at least one pass
    int bits = 0;
    while (bits < 32 && ((int64_t)1 << bits) < K) ++bits;
    const int passes = std::max(1, (bits + 7) / 8);
    const int64_t T = (nnz + kRTile - 1) / kRTile;
    const int64_t nh = (int64_t)kRBins * T;

    uint32_t *kbuf[2] = {nullptr, nullptr};
    int32_t *vbuf[2] = {nullptr, nullptr};
    int32_t *row_of = nullptr;
    int *hist = nullptr, *offs = nullptr, *bsum = nullptr;
    const size_t ebytes = sizeof(int32_t) * (size_t)nnz;
    e = t_alloc((void **)&kbuf[0], ebytes);
    if (e == cudaSuccess) e = t_alloc((void **)&kbuf[1], ebytes);
    if (e == cudaSuccess) e = t_alloc((void **)&vbuf[0], ebytes);
    if (e == cudaSuccess) e = t_alloc((void **)&vbuf[1], ebytes);
    if (e == cudaSuccess) e = t_alloc((void **)&row_of, ebytes);
    if (e == cudaSuccess) e = t_alloc((void **)&hist, sizeof(int) * (size_t)nh);
    if (e == cudaSuccess) e = t_alloc((void **)&offs, sizeof(int) * (size_t)nh);
    if (e == cudaSuccess)
        e = t_alloc((void **)&bsum, sizeof(int) * (size_t)((nh + kScanThreads - 1) / kScanThreads));

    const uint32_t *kin = reinterpret_cast<const uint32_t *>(col);
    const int32_t *vin = nullptr;   // the first pass ranks entry indices
    int cur = 0;
    for (int pass = 0; pass < passes && e == cudaSuccess; ++pass) {
        const int shift = 8 * pass;
        k_radix_hist<<<(unsigned)T, kRThreads, 0, s>>>(kin, nnz, shift, T, hist);
        count_launch();
        e = cudaGetLastError();
        if (e == cudaSuccess) e = device_scan(hist, offs, nh, bsum, s);
        if (e == cudaSuccess) {
            k_radix_scatter<<<(unsigned)T, kRThreads, 0, s>>>(kin, vin, kbuf[cur], vbuf[cur], nnz,
                                                              shift, T, offs);
            count_launch();
            e = cudaGetLastError();
        }
        kin = kbuf[cur];
        vin = vbuf[cur];
        cur ^= 1;
    }
    if (e == cudaSuccess) {
        k_row_of<<<(unsigned)grid_for(p->M * 32, 256, sms), 256, 0, s>>>(p->rowptr, p->M, row_of);
        k_gather_t<<<(unsigned)grid_for(nnz, 256, sms), 256, 0, s>>>(
            vin, row_of, p->rowptr, val, nnz, scale_mean ? 1 : 0, colT, valT);
        k_bounds<<<(unsigned)grid_for(K + 1, 256, sms), 256, 0, s>>>(kin, nnz, K, rowptrT);
        count_launch(3);
        e = cudaGetLastError();
    }
    const cudaError_t es = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = es;
    for (void *q : {(void *)kbuf[0], (void *)kbuf[1], (void *)vbuf[0], (void *)vbuf[1],
                    (void *)row_of, (void *)hist, (void *)offs, (void *)bsum})
        if (q) cudaFree(q);
    return t_status(e);
}

spmm_status spmm_maxpool_backward(spmm_plan_t planT, const int32_t *colT, const float *valT,
                                  const float *B, const int32_t *argmax, const float *dC,
                                  int64_t N, float *dB, void *stream) {
    using namespace spmm;
    if (!planT || N < 0) return SPMM_ERR_INVALID_ARG;
    const Plan *p = reinterpret_cast<const Plan *>(planT);
    const int64_t rows = p->M;
    if (rows == 0 || N == 0) return SPMM_OK;
    if (!dB) return SPMM_ERR_INVALID_ARG;
    if (p->nnz > 0 && (!colT || !argmax || !dC)) return SPMM_ERR_INVALID_ARG;
    if (p->nnz > 0 && valT && !B) return SPMM_ERR_INVALID_ARG;
    if (N >= INT32_MAX / 4) return SPMM_ERR_UNSUPPORTED;
    const bool v4 = N % 4 == 0 && (uintptr_t)dC % 16 == 0 && (uintptr_t)argmax % 16 == 0 &&
                    (uintptr_t)dB % 16 == 0 && (uintptr_t)B % 16 == 0;
    const int V = v4 ? 4 : 1;
    int lanes = 1;
    while (lanes < 32 && (int64_t)lanes * V < N) lanes <<= 1;
    const int64_t rows_per_block = (256 / 32) * (32 / lanes);
    const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    cudaStream_t s = (cudaStream_t)stream;
    const bool hv = valT != nullptr;
    Plan *pm = const_cast<Plan *>(p);
    if (p->n_heavy > 0) {
        const spmm_status st = plan_ensure_workspace(pm, (size_t)p->n_chunks * (size_t)N * 4);
        if (st != SPMM_OK) return st;
    }
    const int ts = (int)std::min<int64_t>(p->t_split, INT32_MAX);
    if (v4) {
        if (hv) k_maxpool_bwd<4, true><<<(unsigned)blocks, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, rows, N, lanes, ts, dB);
        else k_maxpool_bwd<4, false><<<(unsigned)blocks, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, rows, N, lanes, ts, dB);
    } else {
        if (hv) k_maxpool_bwd<1, true><<<(unsigned)blocks, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, rows, N, lanes, ts, dB);
        else k_maxpool_bwd<1, false><<<(unsigned)blocks, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, rows, N, lanes, ts, dB);
    }
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && p->n_heavy > 0) {
        float *ws = reinterpret_cast<float *>(pm->work);
        const unsigned cb = (unsigned)((p->n_chunks + 7) / 8), hb = (unsigned)((p->n_heavy + 7) / 8);
        const int ch = (int)p->chunk;
        if (v4) {
            if (hv) k_maxpool_chunks<4, true><<<cb, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, N, p->chunks, p->n_chunks, ch, ws);
            else k_maxpool_chunks<4, false><<<cb, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, N, p->chunks, p->n_chunks, ch, ws);
            k_maxpool_combine<4><<<hb, 256, 0, s>>>(p->heavy_rows, p->heavy_chunk0, p->n_heavy, N, ws, dB);
        } else {
            if (hv) k_maxpool_chunks<1, true><<<cb, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, N, p->chunks, p->n_chunks, ch, ws);
            else k_maxpool_chunks<1, false><<<cb, 256, 0, s>>>(p->rowptr, colT, valT, B, argmax, dC, N, p->chunks, p->n_chunks, ch, ws);
            k_maxpool_combine<1><<<hb, 256, 0, s>>>(p->heavy_rows, p->heavy_chunk0, p->n_heavy, N, ws, dB);
        }
        count_launch(2);
        e = cudaGetLastError();
    }
    return t_status(e);
}

}  // extern "C"
