// spmm_run_noalloc: the CSR SpMM of spmm_run without a plan and without any
// device allocation, for callers that cannot allocate device memory.
//
// The scratch the long-row split needs (heavy-row list, chunk table, chunk
// partials) lives in one file-scope device array of kStaticScratchBytes. Every
// GPU that loads this library holds that array until the process exits. Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore come before any
// stream capture.
//
// All calls share the one array, which keeps the contents of the last call:
// calls whose GPU work overlaps (two streams, or two host threads) race on it
// and must be serialised by the caller. Every value a call reads from the
// array is written earlier by the same call (the counts are reset by the
// kernel that builds them), so nothing has to start at zero.
#include <mutex>

#include "common.cuh"

namespace spmm {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kNaMaxHeavy = 1 << 16;                        // split rows per call
constexpr int kNaMaxChunks = 1 << 18;                       // chunks per call
constexpr int kNaMaxDevices = 64;

// layout of the array (bytes)
constexpr int kNaMaxBlocks = 1 << 16;                               // row blocks per call
constexpr size_t kNaOffHeader = 0;                                   // int32 [16]
constexpr size_t kNaOffBlocks = 256;                                 // int4 [kNaMaxBlocks]
constexpr size_t kNaOffRows = kNaOffBlocks + 16 * size_t(kNaMaxBlocks); // int32 [kNaMaxHeavy]
constexpr size_t kNaOffChunk0 = kNaOffRows + 4 * size_t(kNaMaxHeavy);  // int32 [kNaMaxHeavy + 1]
constexpr size_t kNaOffChunks =
    (kNaOffChunk0 + 4 * size_t(kNaMaxHeavy + 1) + 255) / 256 * 256;   // int2 [kNaMaxChunks]
constexpr size_t kNaOffPartials =
    (kNaOffChunks + 8 * size_t(kNaMaxChunks) + 255) / 256 * 256;      // fp32 (+ int32 for max)
constexpr size_t kNaPartialBytes = kStaticScratchBytes - kNaOffPartials;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

namespace {

constexpr int kNaThreads = 256;

// The split rows (above t_split) and their chunk counts, in three passes over
// row blocks of `rpb` rows: (1) per block, the split rows, their chunks and
// any decreasing row pointer; (2) one CTA turns the counts into each block's
// first list position and first chunk (exclusive scans, in block order) and
// writes the header: [0] split rows, [1] chunks, [2] table overflow,
// [3] decreasing rowptr; (3) per block, its split rows in row order with the
// index of their first chunk (ceil(d / chunk) chunks each).
__device__ __forceinline__ int na_chunks(int d, int t_split, int chunk) {
    return d > t_split ? (d + chunk - 1) / chunk : 0;
}

__global__ void __launch_bounds__(kNaThreads) k_na_count(const int32_t *__restrict__ rowptr,
                                                         int64_t M, int64_t rpb, int t_split,
                                                         int chunk, int4 *__restrict__ blocks) {
    const int64_t r0 = (int64_t)blockIdx.x * rpb, r1 = min(M, r0 + rpb);
    int heavy = 0, chunks = 0, bad = 0;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += kNaThreads) {
        const int d = rowptr[r + 1] - rowptr[r];
        bad |= d < 0;
        heavy += d > t_split;
        chunks += na_chunks(d, t_split, chunk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        heavy += __shfl_xor_sync(0xffffffffu, heavy, o);
        chunks += __shfl_xor_sync(0xffffffffu, chunks, o);
    }
    bad = __syncthreads_or(bad);
    __shared__ int sh[2][kNaThreads / 32];
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sh[0][w] = heavy;
        sh[1][w] = chunks;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int h = 0, c = 0;
        for (int i = 0; i < kNaThreads / 32; ++i) {
            h += sh[0][i];
            c += sh[1][i];
        }
        blocks[blockIdx.x] = make_int4(h, c, bad, 0);
    }
}

__global__ void __launch_bounds__(1024) k_na_scan(int4 *__restrict__ blocks, int64_t nblk,
                                                  int32_t *__restrict__ hdr) {
    __shared__ int s_h[32], s_c[32];
    __shared__ int s_bh, s_bc, s_bad;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        s_bh = 0;
        s_bc = 0;
        s_bad = 0;
    }
    __syncthreads();
    for (int64_t base = 0; base < nblk; base += 1024) {
        const int64_t b = base + threadIdx.x;
        int4 v = b < nblk ? blocks[b] : make_int4(0, 0, 0, 0);
        int h = v.x, c = v.y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {       // inclusive warp scans
            const int th = __shfl_up_sync(0xffffffffu, h, o), tc = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) { h += th; c += tc; }
        }
        if (lane == 31) { s_h[w] = h; s_c[w] = c; }
        if (v.z) atomicOr(&s_bad, 1);
        __syncthreads();
        int hb = s_bh, cb = s_bc, ht = 0, ct = 0;
        for (int i = 0; i < 32; ++i) {
            if (i < w) { hb += s_h[i]; cb += s_c[i]; }
            ht += s_h[i];
            ct += s_c[i];
        }
        if (b < nblk) blocks[b] = make_int4(hb + h - v.x, cb + c - v.y, v.z, 0);
        __syncthreads();
        if (threadIdx.x == 0) { s_bh += ht; s_bc += ct; }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        hdr[0] = s_bh;
        hdr[1] = s_bc;
        hdr[2] = (s_bh > kNaMaxHeavy || s_bc > kNaMaxChunks) ? 1 : 0;
        hdr[3] = s_bad;
    }
}

__global__ void __launch_bounds__(kNaThreads) k_na_list(const int32_t *__restrict__ rowptr,
                                                        int64_t M, int64_t rpb, int t_split,
                                                        int chunk, const int4 *__restrict__ blocks,
                                                        const int32_t *__restrict__ hdr,
                                                        int32_t *__restrict__ rows,
                                                        int32_t *__restrict__ chunk0) {
    __shared__ int s_cnt[kNaThreads / 32], s_q[kNaThreads / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t r0 = (int64_t)blockIdx.x * rpb, r1 = min(M, r0 + rpb);
    const int4 off = blocks[blockIdx.x];
    int base = off.x, cbase = off.y;
    for (int64_t rb = r0; rb < r1; rb += kNaThreads) {
        const int64_t r = rb + threadIdx.x;
        const int d = r < r1 ? rowptr[r + 1] - rowptr[r] : 0;
        const bool heavy = d > t_split;
        const int q = na_chunks(d, t_split, chunk);
        const unsigned m = __ballot_sync(0xffffffffu, heavy);
        int qs = q;                               // inclusive scan of chunk counts in the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tq = __shfl_up_sync(0xffffffffu, qs, o);
            if (lane >= o) qs += tq;
        }
        if (lane == 31) { s_cnt[w] = __popc(m); s_q[w] = qs; }
        __syncthreads();
        int before = 0, qbefore = 0, tot = 0, qtot = 0;
        for (int i = 0; i < kNaThreads / 32; ++i) {
            if (i < w) { before += s_cnt[i]; qbefore += s_q[i]; }
            tot += s_cnt[i];
            qtot += s_q[i];
        }
        if (heavy) {
            const int pos = base + before + __popc(m & ((1u << lane) - 1u));
            if (pos < kNaMaxHeavy) {
                rows[pos] = (int32_t)r;
                chunk0[pos] = cbase + qbefore + qs - q;
            }
        }
        base += tot;
        cbase += qtot;
        __syncthreads();
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0 && hdr[0] <= kNaMaxHeavy)
        chunk0[hdr[0]] = hdr[1];
}

// One warp per split row writes the (row, first entry) pair of each chunk.
__global__ void k_na_chunks(const int32_t *__restrict__ rowptr, int n_heavy, int chunk,
                            const int32_t *__restrict__ rows, const int32_t *__restrict__ chunk0,
                            int2 *__restrict__ chunks) {
    const int64_t h = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (h >= n_heavy) return;
    const int row = rows[h];
    const int c0 = chunk0[h], c1 = chunk0[h + 1];
    const int b = rowptr[row];
    for (int q = c0 + lane; q < c1; q += 32) chunks[q] = make_int2(row, b + (q - c0) * chunk);
}

std::mutex g_na_mu;
void *g_na_ptr[kNaMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
cudaError_t scratch_address(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_na_ptr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_na_ptr[dev]);
    return cudaSuccess;
}

spmm_status na_status(cudaError_t e) {
    return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
}

int64_t pow2_at_least(int64_t x) {
    int64_t p = 1;
    while (p < x) p <<= 1;
    return p;
}

}  // namespace
}  // namespace spmm

using namespace spmm;

extern "C" spmm_status spmm_run_noalloc(const int32_t *rowptr, const int32_t *col,
                                        const float *val, const float *B, int64_t M, int64_t K,
                                        int64_t N, spmm_reduce reduce, float *C, int32_t *argmax,
                                        void *stream) {
    if (M < 0 || K < 0 || N < 0 || reduce < SPMM_SUM || reduce > SPMM_MAX) return SPMM_ERR_INVALID_ARG;
    if (M >= INT32_MAX || K >= INT32_MAX || N >= INT32_MAX / 4) return SPMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SPMM_OK;
    if (!rowptr || !C) return SPMM_ERR_INVALID_ARG;
    if (reduce != SPMM_MAX) argmax = nullptr;
    cudaStream_t s = (cudaStream_t)stream;

    int dev = 0, num_sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_status(e);
    if (dev < 0 || dev >= kNaMaxDevices) return SPMM_ERR_UNSUPPORTED;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return na_status(e);
    unsigned char *scratch = nullptr;
    e = scratch_address(dev, &scratch);
    if (e != cudaSuccess) return na_status(e);
    int32_t *hdr = reinterpret_cast<int32_t *>(scratch + kNaOffHeader);
    int32_t *rows = reinterpret_cast<int32_t *>(scratch + kNaOffRows);
    int32_t *chunk0 = reinterpret_cast<int32_t *>(scratch + kNaOffChunk0);
    int2 *chunks = reinterpret_cast<int2 *>(scratch + kNaOffChunks);
    float *partials = reinterpret_cast<float *>(scratch + kNaOffPartials);

    // nnz and rowptr[0] (a 4-byte read each; the stream is drained here)
    int32_t ends[2] = {0, 0};
    e = cudaMemcpyAsync(&ends[0], rowptr, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&ends[1], rowptr + M, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return na_status(e);
    if (ends[0] != 0 || ends[1] < 0) return SPMM_ERR_INVALID_INPUT;
    const int64_t nnz = ends[1];
    if (nnz > INT32_MAX - 64) return SPMM_ERR_UNSUPPORTED;
    if (nnz > 0 && (!col || !B)) return SPMM_ERR_INVALID_ARG;

    // split rows and their chunk table, counted on the device and read back
    const int64_t t_split = spmm_default_t_split(M, nnz, num_sms);
    const int64_t chunk = std::max<int64_t>(32, t_split / 2);
    const int64_t rpb = std::max<int64_t>(4096, (M + kNaMaxBlocks - 1) / kNaMaxBlocks);
    const int64_t nblk = (M + rpb - 1) / rpb;
    int4 *blocks = reinterpret_cast<int4 *>(scratch + kNaOffBlocks);
    k_na_count<<<(unsigned)nblk, kNaThreads, 0, s>>>(rowptr, M, rpb, (int)t_split, (int)chunk,
                                                     blocks);
    k_na_scan<<<1, 1024, 0, s>>>(blocks, nblk, hdr);
    k_na_list<<<(unsigned)nblk, kNaThreads, 0, s>>>(rowptr, M, rpb, (int)t_split, (int)chunk,
                                                    blocks, hdr, rows, chunk0);
    count_launch(3);
    int32_t h[4] = {0, 0, 0, 0};
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(h, hdr, sizeof(h), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return na_status(e);
    if (h[3]) return SPMM_ERR_INVALID_INPUT;
    const int64_t n_heavy = h[0], n_chunks = h[1];
    const size_t part_bytes = (size_t)n_chunks * (size_t)N * 4 * (reduce == SPMM_MAX ? 2 : 1);
    if (h[2] || part_bytes > kNaPartialBytes) return SPMM_ERR_UNSUPPORTED;   // beyond the array
    if (n_heavy > 0) {
        const int64_t blocks = (n_heavy + 7) / 8;
        k_na_chunks<<<(unsigned)blocks, 256, 0, s>>>(rowptr, (int)n_heavy, (int)chunk, rows,
                                                     chunk0, chunks);
        count_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return na_status(e);
    }

    // the product: WARPROW for rows up to t_split, the two-phase split for the rest
    const bool aligned = ((uintptr_t)B % 16 == 0) && ((uintptr_t)C % 16 == 0) &&
                         ((uintptr_t)argmax % 16 == 0);
    const int vec = (aligned && N % 4 == 0) ? 4 : 1;
    const int64_t n_vec = (N + vec - 1) / vec;
    const int64_t lanes = std::min<int64_t>(32, std::max<int64_t>(2, pow2_at_least(n_vec)));
    const int64_t tiles = std::max<int64_t>(1, (n_vec + lanes - 1) / lanes);
    if (tiles > kMaxTilesY) return SPMM_ERR_UNSUPPORTED;
    RunArgs a{};
    a.rowptr = rowptr;
    a.col = col;
    a.val = val;
    a.B = B;
    a.C = C;
    a.argmax = argmax;
    a.M = M;
    a.K = K;
    a.nnz4 = (int32_t)(nnz & ~(int64_t)3);
    a.N = (int32_t)N;
    a.n_vec = (int32_t)n_vec;
    a.t_split = (int32_t)t_split;
    a.chunk = (int32_t)chunk;
    a.n_chunks = (int32_t)n_chunks;
    a.n_heavy = (int32_t)n_heavy;
    a.chunks = chunks;
    a.heavy_rows = rows;
    a.heavy_chunk0 = chunk0;
    a.ws_val = partials;
    a.ws_arg = reduce == SPMM_MAX
                   ? reinterpret_cast<int32_t *>(scratch + kNaOffPartials +
                                                 (size_t)n_chunks * (size_t)N * 4)
                   : nullptr;
    a.err = hdr + 8;
    const bool has_val = val != nullptr;
    e = launch_warprow(a, vec, (int)lanes, reduce, has_val, (int)tiles, s);
    if (e == cudaSuccess && n_heavy > 0)
        e = launch_heavy(a, vec, (int)lanes, reduce, has_val, (int)tiles, s);
    return na_status(e);
}
