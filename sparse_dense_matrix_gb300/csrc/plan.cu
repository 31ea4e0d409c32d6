// The C ABI: plan creation (descriptors, heavy-row tables), the router,
// spmm_run's dispatch, validation and status reporting.
//
// Plan creation is one O(M) pass over rowptr on the device (RA-SpMM abstract
// and "routing rules": M, mean degree d = nnz/M and the degree coefficient of
// variation CV_d from the row-pointer array alone), plus an ordered compaction
// of the heavy rows. Integer sums are exact (64-bit), so the descriptors and
// every routing decision are deterministic.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cmath>
#include <new>
#include <vector>

#include "common.cuh"

namespace spmm {

std::atomic<uint64_t> g_launches{0};

namespace {

constexpr int kDescThreads = 256;
constexpr int kDescRowsPerBlock = 4096;

struct BlockStats {
    unsigned long long s1, s2;   // sum of degrees, sum of squared degrees
    int dmax, n_empty, n_bad, n_heavy;
};

// ---------------------------------------------------------------- allocation
// Host-side fault injection for the tests: SPMM_FAULT_ALLOC=n makes the n-th
// device allocation of a spmm_plan_create call fail (as if the device were full).
thread_local int t_alloc_countdown = 0;

cudaError_t dev_alloc(void **p, size_t bytes) {
    *p = nullptr;
    if (t_alloc_countdown > 0 && --t_alloc_countdown == 0) return cudaErrorMemoryAllocation;
    if (bytes == 0) bytes = 16;
    return cudaMalloc(p, bytes);
}

void dev_free(void *p) {
    if (p) cudaFree(p);
}

spmm_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SPMM_OK;
    if (e == cudaErrorMemoryAllocation) return SPMM_ERR_OOM;
    return SPMM_ERR_CUDA;
}

// ------------------------------------------------------------ device kernels
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ int warp_max_i(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// A row-range plan's copy of rowptr starts at the range's first entry:
// subtract it so that the copy is a CSR row-pointer array of its own.
__global__ void k_rebase(int32_t *__restrict__ rp, int64_t n, int32_t base) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        rp[i] -= base;
}

// Block b summarises rows [b*R, (b+1)*R): degree sums, max, empty rows,
// decreasing row pointers, rows above t_split.
__global__ void __launch_bounds__(kDescThreads) k_desc(const int32_t *__restrict__ rowptr,
                                                      int64_t M, int64_t t_split,
                                                      BlockStats *__restrict__ out) {
    const int64_t r0 = (int64_t)blockIdx.x * kDescRowsPerBlock;
    const int64_t r1 = min(M, r0 + kDescRowsPerBlock);
    unsigned long long s1 = 0, s2 = 0;
    int dmax = 0, n_empty = 0, n_bad = 0, n_heavy = 0;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += kDescThreads) {
        const int d = rowptr[r + 1] - rowptr[r];
        if (d < 0) { ++n_bad; continue; }
        s1 += (unsigned long long)d;
        s2 += (unsigned long long)d * (unsigned long long)d;
        dmax = max(dmax, d);
        n_empty += (d == 0);
        n_heavy += (d > t_split);
    }
    s1 = warp_sum_u64(s1);
    s2 = warp_sum_u64(s2);
    dmax = warp_max_i(dmax);
    n_empty = warp_sum_i(n_empty);
    n_bad = warp_sum_i(n_bad);
    n_heavy = warp_sum_i(n_heavy);
    __shared__ BlockStats sh[kDescThreads / kWarp];
    const int w = threadIdx.x / kWarp;
    if ((threadIdx.x & 31) == 0) sh[w] = BlockStats{s1, s2, dmax, n_empty, n_bad, n_heavy};
    __syncthreads();
    if (threadIdx.x == 0) {
        BlockStats t = sh[0];
        for (int i = 1; i < kDescThreads / kWarp; ++i) {
            t.s1 += sh[i].s1;
            t.s2 += sh[i].s2;
            t.dmax = max(t.dmax, sh[i].dmax);
            t.n_empty += sh[i].n_empty;
            t.n_bad += sh[i].n_bad;
            t.n_heavy += sh[i].n_heavy;
        }
        out[blockIdx.x] = t;
    }
}

// Ordered compaction of the heavy rows of block b's row range to offset[b]:
// rows are taken in rounds of kDescThreads consecutive rows, ranked by warp
// ballots and a scan over the warps.
__global__ void __launch_bounds__(kDescThreads) k_heavy_list(const int32_t *__restrict__ rowptr,
                                                            int64_t M, int64_t t_split,
                                                            const int32_t *__restrict__ offset,
                                                            int32_t *__restrict__ heavy_rows,
                                                            int2 *__restrict__ heavy_span) {
    constexpr int kWarps = kDescThreads / kWarp;
    __shared__ int warp_count[kWarps];
    const int64_t r0 = (int64_t)blockIdx.x * kDescRowsPerBlock;
    const int64_t r1 = min(M, r0 + kDescRowsPerBlock);
    const int lane = threadIdx.x & 31, w = threadIdx.x / kWarp;
    int base = offset[blockIdx.x];
    for (int64_t rb = r0; rb < r1; rb += kDescThreads) {
        const int64_t r = rb + threadIdx.x;
        int b = 0, e = 0;
        bool heavy = false;
        if (r < r1) {
            b = rowptr[r];
            e = rowptr[r + 1];
            heavy = (e - b) > t_split;
        }
        const unsigned m = __ballot_sync(0xffffffffu, heavy);
        if (lane == 0) warp_count[w] = __popc(m);
        __syncthreads();
        int before = 0, total = 0;
        for (int i = 0; i < kWarps; ++i) {
            before += (i < w) ? warp_count[i] : 0;
            total += warp_count[i];
        }
        if (heavy) {
            const int pos = base + before + __popc(m & ((1u << lane) - 1u));
            heavy_rows[pos] = (int)r;
            heavy_span[pos] = make_int2(b, e);
        }
        base += total;
        __syncthreads();
    }
}

// Column check and column-spread histogram, one warp per row: every entry must
// satisfy 0 <= col < K; |col - row| is binned by b = ceil(log2 |col - row|)
// (b = 0 for distances 0 and 1). Warp-aggregated shared-memory counters, one
// global add per bin per block (integer counts: the result is exact).
constexpr int kSpreadBins = 34;
// two more counters after the spread bins: entries inside their row's diagonal
// block of kBlockRows x kBlockRows (col / kBlockRows == row / kBlockRows), and
// entries whose column is below the previous entry's in the same row
constexpr int kHistWords = kSpreadBins + 2;
// Rows are local to the plan; the spread and the diagonal blocks are measured
// against the global row (row + row0) that a row-range plan's row stands for.
// A warp takes one work item: a row of at most t_split entries, or one chunk
// of a longer row from the plan's chunk table, so that no warp walks a hub
// row of ~1e5 entries alone (that tail had set the pass's time).
__global__ void __launch_bounds__(256) k_check_cols(const int32_t *__restrict__ rowptr,
                                                   const int32_t *__restrict__ col, int64_t M,
                                                   int64_t K, int64_t row0, int64_t t_split,
                                                   int64_t chunk, const int2 *__restrict__ chunks,
                                                   int64_t n_chunks, int32_t *__restrict__ err,
                                                   unsigned long long *__restrict__ hist) {
    __shared__ unsigned int sh[kHistWords];
    for (int b = threadIdx.x; b < kHistWords; b += blockDim.x) sh[b] = 0;
    __syncthreads();
    int bad = 0;
    const int lane = threadIdx.x & 31;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
         item < M + n_chunks; item += warps) {
        int64_t row;
        int p0, pa, p1;      // row start (for the order check), then the item's entries [pa, p1)
        if (item < M) {
            row = item;
            p0 = rowptr[row];
            p1 = rowptr[row + 1];
            if (p1 - p0 > t_split) continue;            // uniform per warp: chunked below
            pa = p0;
        } else {
            const int2 ch = chunks[item - M];
            row = ch.x;
            pa = ch.y;
            p0 = rowptr[row];
            p1 = (int)min((int64_t)pa + chunk, (int64_t)rowptr[row + 1]);
        }
        for (int pb = pa; pb < p1; pb += 32) {
            const int p = pb + lane;
            int b = -1;
            bool in_blk = false, descent = false;
            if (p < p1) {
                const int c = col[p];
                descent = p > p0 && c < col[p - 1];
                if (c < 0 || (int64_t)c >= K) {
                    bad = 1;
                } else {
                    const int64_t g = row + row0;
                    const unsigned long long dist =
                        (unsigned long long)((int64_t)c > g ? (int64_t)c - g : g - (int64_t)c);
                    b = dist <= 1 ? 0 : 64 - __clzll((long long)(dist - 1));
                    in_blk = ((int64_t)c / kBlockRows) == (g / kBlockRows);
                }
            }
            const unsigned peers = __match_any_sync(__activemask(), b);
            if (b >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh[b], (unsigned)__popc(peers));
            const unsigned nb = __popc(__ballot_sync(__activemask(), in_blk));
            if (lane == 0 && nb) atomicAdd(&sh[kSpreadBins], nb);
            const unsigned nd = __popc(__ballot_sync(__activemask(), descent));
            if (lane == 0 && nd) atomicAdd(&sh[kSpreadBins + 1], nd);
        }
    }
    __syncthreads();
    for (int b = threadIdx.x; b < kHistWords; b += blockDim.x)
        if (sh[b]) atomicAdd(&hist[b], (unsigned long long)sh[b]);
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err + kErrBadCol, 1);
}

// SEGMENT tiles: tile t starts at merge-path item k = t * kSegItems (items are
// the row ends and the stored entries, a row's end after its entries). After k
// items the path has passed r row ends, r the largest row index with
// rowptr[r] + r <= k (rowptr[r] + r strictly increases with r), and
// e = k - r entries. One thread per tile boundary, a binary search each.
__global__ void k_seg_tiles(const int32_t *__restrict__ rowptr, int64_t M, int64_t items,
                            int64_t n_tiles, int2 *__restrict__ out) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t <= n_tiles;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = min(t * (int64_t)kSegItems, items);
        int64_t lo = 0, hi = M;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if ((int64_t)rowptr[mid] + mid <= k) lo = mid;
            else hi = mid - 1;
        }
        out[t] = make_int2((int)lo, (int)(k - lo));
    }
}

// ------------------------------------------------------------- host helpers
int64_t pow2ceil(int64_t x) {
    int64_t p = 1;
    while (p < x) p <<= 1;
    return p;
}

void free_heavy(Plan *p) {
    dev_free(p->heavy_rows);
    dev_free(p->heavy_chunk0);
    dev_free(p->chunks);
    p->heavy_rows = nullptr;
    p->heavy_chunk0 = nullptr;
    p->chunks = nullptr;
    p->n_heavy = p->n_chunks = 0;
}

// Descriptors, validation and heavy-row tables for threshold t_split.
spmm_status analyse(Plan *p, int64_t t_split, cudaStream_t s) {
    free_heavy(p);
    p->t_split = t_split;
    p->chunk = std::max<int64_t>(32, t_split / 2);
    if (p->M == 0) return SPMM_OK;
    const int64_t nblk = (p->M + kDescRowsPerBlock - 1) / kDescRowsPerBlock;
    BlockStats *d_stats = nullptr;
    int32_t *d_off = nullptr;
    int2 *d_span = nullptr;
    spmm_status st = SPMM_OK;
    std::vector<BlockStats> hs(nblk);
    std::vector<int32_t> off(nblk + 1, 0);
    cudaError_t e = dev_alloc((void **)&d_stats, sizeof(BlockStats) * nblk);
    if (e != cudaSuccess) return from_cuda(e);
    k_desc<<<(unsigned)nblk, kDescThreads, 0, s>>>(p->rowptr, p->M, t_split, d_stats);
    count_launch();
    e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(hs.data(), d_stats, sizeof(BlockStats) * nblk, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) { st = from_cuda(e); goto done; }
    {
        unsigned long long s1 = 0, s2 = 0;
        int64_t dmax = 0, empty = 0, bad = 0, heavy = 0;
        for (int64_t b = 0; b < nblk; ++b) {
            s1 += hs[b].s1;
            s2 += hs[b].s2;
            dmax = std::max<int64_t>(dmax, hs[b].dmax);
            empty += hs[b].n_empty;
            bad += hs[b].n_bad;
            off[b] = (int32_t)heavy;
            heavy += hs[b].n_heavy;
        }
        off[nblk] = (int32_t)heavy;
        if (bad || (int64_t)s1 != p->nnz) { st = SPMM_ERR_INVALID_INPUT; goto done; }
        p->d_max = dmax;
        p->n_empty = empty;
        p->dbar = (double)s1 / (double)p->M;
        const double var = (double)s2 / (double)p->M - p->dbar * p->dbar;
        p->cv = s1 == 0 ? 0.0 : std::sqrt(var > 0.0 ? var : 0.0) / p->dbar;
        p->n_heavy = heavy;
    }
    if (p->n_heavy > 0) {
        const int64_t nh = p->n_heavy;
        e = dev_alloc((void **)&d_off, sizeof(int32_t) * (nblk + 1));
        if (e == cudaSuccess) e = dev_alloc((void **)&p->heavy_rows, sizeof(int32_t) * nh);
        if (e == cudaSuccess) e = dev_alloc((void **)&d_span, sizeof(int2) * nh);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d_off, off.data(), sizeof(int32_t) * (nblk + 1), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) {
            k_heavy_list<<<(unsigned)nblk, kDescThreads, 0, s>>>(p->rowptr, p->M, t_split, d_off,
                                                                 p->heavy_rows, d_span);
            count_launch();
            e = cudaGetLastError();
        }
        std::vector<int2> span(nh);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(span.data(), d_span, sizeof(int2) * nh, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) { st = from_cuda(e); goto done; }
        // chunk table: heavy row h is cut into ceil(d_h / chunk) chunks
        std::vector<int32_t> c0(nh + 1, 0);
        std::vector<int2> chunks;
        std::vector<int32_t> rows(nh);
        e = cudaMemcpy(rows.data(), p->heavy_rows, sizeof(int32_t) * nh, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) { st = from_cuda(e); goto done; }
        for (int64_t h = 0; h < nh; ++h) {
            c0[h] = (int32_t)chunks.size();
            for (int64_t q = span[h].x; q < span[h].y; q += p->chunk)
                chunks.push_back(make_int2(rows[h], (int)q));
        }
        c0[nh] = (int32_t)chunks.size();
        p->n_chunks = (int64_t)chunks.size();
        e = dev_alloc((void **)&p->heavy_chunk0, sizeof(int32_t) * (nh + 1));
        if (e == cudaSuccess) e = dev_alloc((void **)&p->chunks, sizeof(int2) * p->n_chunks);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(p->heavy_chunk0, c0.data(), sizeof(int32_t) * (nh + 1), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(p->chunks, chunks.data(), sizeof(int2) * p->n_chunks, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) { st = from_cuda(e); goto done; }
    }
done:
    dev_free(d_stats);
    dev_free(d_off);
    dev_free(d_span);
    if (st != SPMM_OK) free_heavy(p);
    return st;
}

void destroy(Plan *p) {
    if (!p) return;
    free_heavy(p);
    block_free(p);
    gather_free(p);
    dev_free(p->seg_tiles);
    dev_free(p->rowptr);
    dev_free(p->work);
    dev_free(p->err);
    delete p;
}

// The SEGMENT family's tile table (see k_seg_tiles).
spmm_status seg_build(Plan *p, cudaStream_t s) {
    const int64_t items = p->M + p->nnz;
    p->seg_n_tiles = (items + kSegItems - 1) / kSegItems;
    cudaError_t e = dev_alloc((void **)&p->seg_tiles, sizeof(int2) * (p->seg_n_tiles + 1));
    if (e != cudaSuccess) return from_cuda(e);
    const int64_t blocks = std::min<int64_t>((p->seg_n_tiles + 256) / 256, 4096);
    k_seg_tiles<<<(unsigned)std::max<int64_t>(1, blocks), 256, 0, s>>>(p->rowptr, p->M, items,
                                                                       p->seg_n_tiles,
                                                                       p->seg_tiles);
    count_launch();
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return from_cuda(e);
}

size_t workspace_need(const Plan *p, int64_t N, int reduce) {
    if (p->n_heavy == 0 || N == 0) return 0;
    const size_t per = (size_t)p->n_chunks * (size_t)N * 4;
    return reduce == SPMM_MAX ? 2 * per : per;
}

spmm_status ensure_workspace(Plan *p, size_t need) {
    if (need <= p->work_bytes) return SPMM_OK;
    dev_free(p->work);
    p->work = nullptr;
    p->work_bytes = 0;
    void *w = nullptr;
    cudaError_t e = cudaMalloc(&w, need);
    if (e != cudaSuccess) return from_cuda(e);
    p->work = w;
    p->work_bytes = need;
    return SPMM_OK;
}

}  // namespace

spmm_status plan_ensure_workspace(Plan *p, size_t need) { return ensure_workspace(p, need); }

// ------------------------------------------------------------------ router
// Rules, first match wins (RA-SpMM "routing rules": descriptors + N -> family):
//   R0  a family pinned by spmm_plan_set_family is used as given (WINDOW only
//       where its conditions hold);
//   R1  column locality (>= 97% of entries within |col - row| <= W, W <= 4096,
//       mean degree >= 2; an out-of-window gather stalls its whole batch),
//       N % 4 == 0 with 16-byte aligned operands, a ring of 3R + 2W B rows
//       that fits in shared memory with at most 4 column tiles,
//       an average tile's entries fitting one pipeline stage (two rows per
//       lane group preferred, else one), a 2W halo at most twice a CTA's
//       row range, and (row-range plans) a first row on a multiple of the
//       tile's R rows                                          -> WINDOW;
//   R1a block-diagonal graphs (>= 85% of the entries in their row's
//       256-column diagonal block, blocks >= 5% dense), sum or mean,
//       N % 16 == 0, aligned B/C, a whole-matrix plan     -> BLOCK (tensor cores);
//   R2  wide N (more than 32 column vectors per row)        -> WARPROW with column
//       tiles (COLTILE, the staged variant, measured 1.1-1.7x slower: pin only);
//   R3  skewed degrees (CV_d > 1), N <= 32 in 128-bit vectors, col/val
//       16-byte aligned                                       -> SEGMENT (merge-path tiles);
//       (GATHER, TMA gather4 of B rows into a shared ring, N % 128 == 0:
//       pin only)
//   R4  near-uniform degrees (CV_d <= 1) and narrow N (L < 32 lanes, so
//       several rows share a warp)                            -> ROWGROUP, 32/L rows per warp;
//   R5  otherwise (skewed degrees)                            -> WARPROW.
// Independently of the family, rows with more than t_split entries are split
// into chunks (two extra launches) whenever the plan holds such rows.
// `aligned`: bit 0 = B/C/argmax 16-byte aligned, bit 1 = col/val 16-byte aligned,
// bit 2 = no val array (unweighted; the WINDOW family then stages no values).
static void route_fill(const spmm_plan_info *d, int64_t N, int reduce, int aligned, int num_sms,
                       int family_override, spmm_plan_info *o) {
    if (o != d) *o = *d;
    o->N = N;
    o->reduce = reduce;
    o->num_sms = num_sms;
    o->window_rows = 0;
    o->window_ctas = 0;
    o->window_smem = 0;
    o->window_chunks = 0;
    o->vec = ((aligned & 1) && N % 4 == 0) ? 4 : 1;
    const int64_t n_vec = (N + o->vec - 1) / o->vec;
    int64_t lanes = std::min<int64_t>(32, std::max<int64_t>(2, pow2ceil(n_vec)));
    int fam = -2;
    // R1: WINDOW
    // (a pinned WINDOW skips the two efficiency conditions: mean degree and halo)
    const bool forced = family_override == SPMM_FAMILY_WINDOW;
    const bool window_ok = (family_override == SPMM_FAMILY_AUTO || forced) &&
                           d->band_w > 0 && (aligned & 3) == 3 && N > 0 && N % 4 == 0 &&
                           (forced || (d->dbar >= 2.0 && d->band_cover >= 0.97)) && d->M > 0;
    // R1a: BLOCK (tensor cores) when pinned, or when at least 85% of the
    // entries lie in their row's 256-column diagonal block and those blocks
    // are at least 5% dense (known after the column check). On the 64k-row
    // community graph (91% of the entries in blocks of density 0.2) it
    // measured 81.9 us at N=128 and 271 us at N=512, against 96.5 and 338 us
    // for WARPROW. Its diagonal blocks are those of a plan that starts at row 0.
    const bool block_shape = d->M > 0 && N > 0 && N % 16 == 0 && (aligned & 1) &&
                             reduce != SPMM_MAX && d->row0 == 0;
    const bool block_dense = d->nnz > 0 && (double)d->blk_intra >= 0.85 * (double)d->nnz &&
                             (double)d->blk_intra >= 0.05 * (double)d->M * kBlockRows;
    if (block_shape && (family_override == SPMM_FAMILY_BLOCK ||
                        (family_override == SPMM_FAMILY_AUTO && block_dense)))
        fam = SPMM_FAMILY_BLOCK;
    int64_t win_tiles = 0;
    if (window_ok && fam == -2) {
        bool found = false;
        // column tiles of cw = 4 L Q columns, widest first: Q = 2 chunks per lane
        // (L = cw / 8) down to cw = 16, then L = 2, Q = 1 for cw = 8
        for (int64_t cw = 4 * std::min<int64_t>(32, std::max<int64_t>(2, pow2ceil((N + 3) / 4)));
             cw >= 8 && !found; cw >>= 1) {
            const int L = cw == 8 ? 2 : cw == 16 ? 4 : (int)(cw / 8);
            const int Q = cw <= 16 ? 1 : 2;
            for (int rpg = 2; rpg >= 1 && !found; --rpg) {
                WinShape w;
                if (!window_shape(d->M, d->K, N, d->dbar, d->band_w, !(aligned & 4), L, Q, rpg,
                                  &w))
                    continue;
                if (w.smem_bytes > kWindowSmemBudget) continue;
                // a row-range plan's tiles must start on whole R-row boxes of B
                if (d->row0 % w.R != 0) continue;
                // the staged entries of an average tile must fit a stage (else the
                // tile is read from global memory)
                if (!forced && (double)w.R * d->dbar * 1.25 + 64 > (double)w.ecap) continue;
                const int64_t tiles_y = (N + cw - 1) / cw;
                if (!forced && tiles_y > 4) continue;
                const int64_t ctas = std::max<int64_t>(
                    1, (num_sms > 0 ? num_sms : 1) * w.ctas_per_sm / tiles_y);
                // the halo rows come from L2 (neighbouring CTAs stream them too):
                // allow a halo up to twice a CTA's own rows
                if (!forced && 2 * d->band_w > 2 * (d->M / ctas)) continue;
                fam = SPMM_FAMILY_WINDOW;
                lanes = L;
                win_tiles = tiles_y;
                o->window_chunks = Q;
                o->window_rows = w.R;
                o->window_ctas = (int32_t)ctas;
                o->window_smem = w.smem_bytes;
                found = true;
            }
        }
    }
    // COLTILE needs 128-bit vectors (N % 4 == 0, aligned B/C); else WARPROW tiles
    const bool coltile_ok = o->vec == 4;
    // SEGMENT needs 128-bit vectors and col/val that bulk copies may read
    // (16-byte aligned)
    const bool segment_ok = o->vec == 4 && (aligned & 2) && d->M > 0 && d->seg_tiles > 0;
    // GATHER needs column tiles of 256 or 128 columns that the gathered rows
    // fill exactly (N % 128 == 0), 16-byte aligned B (its tensor map), C and
    // argmax, and at least one entry
    const bool gather_ok = (aligned & 1) && gather_tile(N) > 0 && d->M > 0 && d->nnz > 0;
    // STREAM needs 128-bit vectors (N % 4 == 0, aligned B/C/argmax), N > 32
    // and at least one entry
    const bool stream_ok = o->vec == 4 && stream_lanes(N) > 0 && d->M > 0 && d->nnz > 0;
    if (fam == -2) {
        if (family_override == SPMM_FAMILY_COLTILE)
            fam = coltile_ok ? SPMM_FAMILY_COLTILE : SPMM_FAMILY_WARPROW;
        else if (family_override == SPMM_FAMILY_SEGMENT)
            fam = segment_ok ? SPMM_FAMILY_SEGMENT : SPMM_FAMILY_WARPROW;
        else if (family_override == SPMM_FAMILY_GATHER)
            fam = gather_ok ? SPMM_FAMILY_GATHER : SPMM_FAMILY_WARPROW;
        else if (family_override == SPMM_FAMILY_STREAM)
            fam = stream_ok ? SPMM_FAMILY_STREAM : SPMM_FAMILY_WARPROW;
        else if (family_override != SPMM_FAMILY_AUTO && family_override != SPMM_FAMILY_WINDOW &&
                 family_override != SPMM_FAMILY_BLOCK)
            fam = family_override;
        else if (n_vec > 32)
            fam = SPMM_FAMILY_WARPROW;   // measured faster than COLTILE on the wide workloads
        else if (segment_ok && d->cv > 1.0 && n_vec <= 8)
            // skewed degrees at narrow N (eight lanes or fewer per entry): the
            // merge-path tiles keep every lane's gathers in flight where a warp
            // per row waits on short rows (Chung-Lu 4M, N=16: 1.37 against
            // 1.71 ms for the sum, 1.81 against 2.24 ms for max; N=32: 2.08
            // against 2.17 ms, 2.70 against 2.99 ms); at N=64 and wider
            // WARPROW measured 8-40% faster
            fam = SPMM_FAMILY_SEGMENT;
        else if (d->cv <= 1.0 && lanes < 32)
            // a 32-lane ROWGROUP holds one row per warp like WARPROW, without
            // WARPROW's batched loads (community graph, N=128: 104 against 94 us)
            fam = SPMM_FAMILY_ROWGROUP;
        else
            fam = SPMM_FAMILY_WARPROW;
    }
    if (fam == SPMM_FAMILY_COLTILE) lanes = 32;     // one 128-column tile per warp
    // SEGMENT: L lanes x Q four-column chunks per lane; two chunks when a row
    // is wider than 128 columns, column tiles of 256 beyond that
    const int64_t seg_q = n_vec > 32 ? 2 : 1;
    if (fam == SPMM_FAMILY_STREAM) lanes = stream_lanes(N);
    o->lanes = (int32_t)lanes;
    if (fam == SPMM_FAMILY_BLOCK || fam == SPMM_FAMILY_GATHER) lanes = 32;
    o->col_tiles = fam == SPMM_FAMILY_WINDOW    ? (int32_t)win_tiles
                   : fam == SPMM_FAMILY_BLOCK   ? (int32_t)((N + 127) / 128)
                   : fam == SPMM_FAMILY_GATHER  ? (int32_t)(N / gather_tile(N))
                   : fam == SPMM_FAMILY_STREAM  ? (int32_t)((n_vec + lanes - 1) / lanes)
                   : fam == SPMM_FAMILY_SEGMENT ? (int32_t)((n_vec + lanes * seg_q - 1) / (lanes * seg_q))
                                                : (int32_t)std::max<int64_t>(1, (n_vec + lanes - 1) / lanes);
    o->family = fam;
    o->rows_per_warp = fam == SPMM_FAMILY_ROWGROUP ? (int32_t)(32 / lanes) : 1;
    o->seg_warps = 0;
    o->seg_chunks = 0;
    o->gather_ctas = 0;
    o->stream_ranges = 0;
    if (fam == SPMM_FAMILY_STREAM) {
        // every row, however long, goes through the entry ranges: no split
        o->stream_ranges = (int32_t)stream_ranges(d->nnz, num_sms, (int)lanes, o->col_tiles);
        o->launches = 2;
        o->workspace_bytes =
            (int64_t)stream_workspace(o->stream_ranges, o->col_tiles, (int)lanes, reduce);
        return;
    }
    if (fam == SPMM_FAMILY_GATHER) {
        // every row, however long, goes through the entry ranges: no split
        o->gather_ctas = (int32_t)gather_ctas(d->nnz, num_sms, o->col_tiles);
        o->launches = 2;
        o->workspace_bytes =
            (int64_t)gather_workspace(o->gather_ctas, o->col_tiles, gather_tile(N), reduce);
        return;
    }
    if (fam == SPMM_FAMILY_BLOCK) {
        // the off-block partial rows, [M][N] fp32
        o->launches = (d->M > 0 && N > 0) ? 1 : 0;
        o->workspace_bytes = d->M * N * 4;
        return;
    }
    if (fam == SPMM_FAMILY_SEGMENT) {
        // every row, however long, goes through the merge-path tiles: no split
        o->seg_chunks = (int32_t)seg_q;
        o->seg_warps = (int32_t)segment_warps(d->seg_tiles, num_sms, o->col_tiles);
        o->launches = (d->M > 0 && N > 0) ? 2 : 0;
        o->workspace_bytes = (int64_t)segment_workspace(o->seg_warps, o->col_tiles, (int)lanes,
                                                        (int)seg_q, reduce);
        return;
    }
    const bool split = d->n_heavy > 0 && fam != SPMM_FAMILY_BLOCK;
    o->launches = (d->M > 0 && N > 0) ? 1 + (split ? 2 : 0) : 0;
    const size_t per = (size_t)d->n_chunks * (size_t)N * 4;
    o->workspace_bytes = split ? (int64_t)(reduce == SPMM_MAX ? 2 * per : per) : 0;
}

}  // namespace spmm

using namespace spmm;

extern "C" {

int64_t spmm_default_t_split(int64_t M, int64_t nnz, int num_sms) {
    (void)M;
    // A row holding more than ~1/128 of one SM's share of the entries would
    // run for a large fraction of the launch on a single warp: split it. On
    // large skewed graphs even rows of a few hundred entries are long next to
    // the median row, so the threshold stops at 512 (measured on the 4M-row
    // Chung-Lu graph: 5388 -> 512 took N=64 from 5.05 to 4.30 ms).
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t share = nnz / (128 * sms);
    return std::min<int64_t>(512, std::max<int64_t>(256, share));
}

spmm_status spmm_route(const spmm_plan_info *desc, int64_t N, spmm_reduce reduce, int aligned,
                       int num_sms, int family_override, spmm_plan_info *out) {
    if (!desc || !out || N < 0) return SPMM_ERR_INVALID_ARG;
    if (reduce < SPMM_SUM || reduce > SPMM_MAX) return SPMM_ERR_INVALID_ARG;
    if (family_override < SPMM_FAMILY_AUTO || family_override > SPMM_FAMILY_STREAM)
        return SPMM_ERR_INVALID_ARG;
    route_fill(desc, N, reduce, aligned, num_sms, family_override, out);
    return SPMM_OK;
}

const char *spmm_status_string(spmm_status s) {
    switch (s) {
        case SPMM_OK: return "ok";
        case SPMM_ERR_INVALID_ARG: return "invalid argument";
        case SPMM_ERR_INVALID_INPUT: return "invalid input (rowptr not a CSR row-pointer array, or a column out of range)";
        case SPMM_ERR_OOM: return "out of memory";
        case SPMM_ERR_CUDA: return "CUDA runtime error";
        case SPMM_ERR_UNSUPPORTED: return "unsupported size";
        case SPMM_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    }
    return "unknown status";
}

uint64_t spmm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Plan over rows [row_begin, row_begin + M) of the CSR array `rowptr`. A whole
// matrix (range == false) must have rowptr[0] == 0; a row range is rebased.
static spmm_status create_plan(const int32_t *rowptr, int64_t row_begin, int64_t M, int64_t K,
                               bool range, void *stream, spmm_plan_t *out) {
    const char *fault = std::getenv("SPMM_FAULT_ALLOC");
    t_alloc_countdown = fault ? std::atoi(fault) : 0;
    cudaStream_t s = (cudaStream_t)stream;
    Plan *p = new (std::nothrow) Plan();
    if (!p) return SPMM_ERR_OOM;
    p->M = M;
    p->K = K;
    spmm_status st = SPMM_OK;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = dev_alloc((void **)&p->rowptr, sizeof(int32_t) * (M + 1 + kRowptrPad));
    if (e == cudaSuccess) e = dev_alloc((void **)&p->err, sizeof(int32_t) * kErrWords);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->err, 0, sizeof(int32_t) * kErrWords, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->rowptr, rowptr + row_begin, sizeof(int32_t) * (M + 1),
                            cudaMemcpyDefault, s);
    int32_t ends[2] = {0, 0};
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ends[0], p->rowptr, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ends[1], p->rowptr + M, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        st = from_cuda(e);
    } else if ((range ? ends[0] < 0 : ends[0] != 0) || ends[1] < ends[0]) {
        st = SPMM_ERR_INVALID_INPUT;
    } else if (ends[1] > INT32_MAX - 64) {
        st = SPMM_ERR_UNSUPPORTED;
    } else {
        p->row0 = row_begin;
        p->col_base = ends[0];
        p->nnz = (int64_t)ends[1] - ends[0];
        if (ends[0] != 0) {
            k_rebase<<<(unsigned)std::min<int64_t>((M + 256) / 256, 4096), 256, 0, s>>>(
                p->rowptr, M + 1, ends[0]);
            count_launch();
            e = cudaGetLastError();
        }
        // pad the copy with rowptr[M] so that tile-sized bulk copies may run past row M
        std::vector<int32_t> pad(kRowptrPad, (int32_t)p->nnz);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(p->rowptr + M + 1, pad.data(), sizeof(int32_t) * kRowptrPad,
                                cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            destroy(p);
            t_alloc_countdown = 0;
            return from_cuda(e);
        }
        p->t_split_default = spmm_default_t_split(M, p->nnz, p->num_sms);
        st = analyse(p, p->t_split_default, s);
        if (st == SPMM_OK && M > 0) st = seg_build(p, s);
    }
    t_alloc_countdown = 0;
    if (st != SPMM_OK) {
        destroy(p);
        return st;
    }
    *out = reinterpret_cast<spmm_plan_t>(p);
    return SPMM_OK;
}

spmm_status spmm_plan_create(const int32_t *rowptr, int64_t M, int64_t K, void *stream,
                             spmm_plan_t *out) {
    if (!out) return SPMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (M < 0 || K < 0 || !rowptr) return SPMM_ERR_INVALID_ARG;
    if (M >= INT32_MAX || K >= INT32_MAX) return SPMM_ERR_UNSUPPORTED;
    return create_plan(rowptr, 0, M, K, false, stream, out);
}

spmm_status spmm_plan_create_range(const int32_t *rowptr, int64_t row_begin, int64_t row_end,
                                   int64_t K, void *stream, spmm_plan_t *out) {
    if (!out) return SPMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (row_begin < 0 || row_end < row_begin || K < 0 || !rowptr) return SPMM_ERR_INVALID_ARG;
    if (row_end >= INT32_MAX || K >= INT32_MAX) return SPMM_ERR_UNSUPPORTED;
    return create_plan(rowptr, row_begin, row_end - row_begin, K, true, stream, out);
}

spmm_status spmm_partition_rows(const int32_t *rowptr, int64_t M, int32_t parts,
                                int64_t align_rows, int64_t *bounds) {
    if (!rowptr || !bounds || M < 0 || parts < 1 || align_rows < 1) return SPMM_ERR_INVALID_ARG;
    if (M >= INT32_MAX) return SPMM_ERR_UNSUPPORTED;
    if (rowptr[0] != 0) return SPMM_ERR_INVALID_INPUT;
    for (int64_t i = 0; i < M; ++i)
        if (rowptr[i + 1] < rowptr[i]) return SPMM_ERR_INVALID_INPUT;
    // work of the rows before row i: their entries plus one per row (its output)
    auto work = [&](int64_t i) { return (int64_t)rowptr[i] + i; };
    const int64_t total = work(M);
    bounds[0] = 0;
    for (int32_t q = 1; q < parts; ++q) {
        const int64_t target = (int64_t)q * total / parts;   // q < 2^31, total < 2^32
        // first row whose prefix work reaches the target
        int64_t lo = 0, hi = M;
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (work(mid) >= target) hi = mid;
            else lo = mid + 1;
        }
        // nearest multiple of align_rows, kept in order and inside [0, M]
        int64_t b = (lo + align_rows / 2) / align_rows * align_rows;
        b = std::min(std::max(b, bounds[q - 1]), M);
        bounds[q] = b;
    }
    bounds[parts] = M;
    return SPMM_OK;
}

spmm_status spmm_plan_destroy(spmm_plan_t plan) {
    destroy(reinterpret_cast<Plan *>(plan));
    return SPMM_OK;
}

static void fill_desc(const Plan *p, spmm_plan_info *o) {
    std::memset(o, 0, sizeof(*o));
    o->M = p->M;
    o->K = p->K;
    o->nnz = p->nnz;
    o->d_max = p->d_max;
    o->n_empty = p->n_empty;
    o->dbar = p->dbar;
    o->cv = p->cv;
    o->t_split = p->t_split;
    o->chunk = p->chunk;
    o->n_heavy = p->n_heavy;
    o->n_chunks = p->n_chunks;
    o->band_w = p->band_w;
    o->rows_sorted = p->rows_sorted ? 1 : 0;
    o->blk_intra = p->blk_intra;
    o->band_cover = p->band_cover;
    o->row0 = p->row0;
    o->seg_tiles = p->seg_n_tiles;
    o->block_bytes = p->bk_bytes;
    o->gather_bytes = p->ga_bytes;
}

spmm_status spmm_plan_describe(spmm_plan_t plan, int64_t N, spmm_reduce reduce, spmm_plan_info *out) {
    if (!plan || !out || N < 0 || reduce < SPMM_SUM || reduce > SPMM_MAX) return SPMM_ERR_INVALID_ARG;
    const Plan *p = reinterpret_cast<const Plan *>(plan);
    fill_desc(p, out);
    route_fill(out, N, reduce, 3, p->num_sms, p->family_override, out);
    return SPMM_OK;
}

spmm_status spmm_plan_set_family(spmm_plan_t plan, int family, int64_t t_split) {
    if (!plan || family < SPMM_FAMILY_AUTO || family > SPMM_FAMILY_STREAM) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    p->family_override = family;
    // The kernels compare row lengths against a 32-bit threshold; no row is
    // longer than INT32_MAX entries, so a larger threshold means the same:
    // split nothing.
    const int64_t want = t_split > 0 ? std::min<int64_t>(t_split, INT32_MAX) : p->t_split_default;
    if (want == p->t_split) return SPMM_OK;
    cudaError_t e = cudaDeviceSynchronize();   // the workspace and tables may be in use
    if (e != cudaSuccess) return from_cuda(e);
    return analyse(p, want, nullptr);
}

spmm_status spmm_plan_reserve(spmm_plan_t plan, int64_t N, spmm_reduce reduce) {
    if (!plan || N < 0 || reduce < SPMM_SUM || reduce > SPMM_MAX) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    // the larger of the split-row partials and the SEGMENT family's open rows
    spmm_plan_info r;
    fill_desc(p, &r);
    route_fill(&r, N, reduce, 7, p->num_sms, SPMM_FAMILY_SEGMENT, &r);
    const size_t seg = r.family == SPMM_FAMILY_SEGMENT ? (size_t)r.workspace_bytes : 0;
    // and the BLOCK family's off-block partial rows when it is the routed family
    fill_desc(p, &r);
    route_fill(&r, N, reduce, 7, p->num_sms, p->family_override, &r);
    const size_t blk = r.family == SPMM_FAMILY_BLOCK ? (size_t)r.workspace_bytes : 0;
    // and the GATHER family's open rows and per-entry row ids when routed
    const bool rows_ids = r.family == SPMM_FAMILY_GATHER || r.family == SPMM_FAMILY_STREAM;
    const size_t gat = rows_ids ? (size_t)r.workspace_bytes : 0;
    if (rows_ids && !p->ga_rid) {
        cudaError_t e = gather_prepare(p, nullptr);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return from_cuda(e);
    }
    return ensure_workspace(
        p, std::max(std::max(workspace_need(p, N, reduce), seg), std::max(blk, gat)));
}

spmm_status spmm_plan_validate_cols(spmm_plan_t plan, const int32_t *col, void *stream) {
    if (!plan) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    if (p->nnz == 0) return SPMM_OK;
    if (!col) return SPMM_ERR_INVALID_ARG;
    col += p->col_base;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t flag = 0;
    unsigned long long *d_hist = nullptr;
    unsigned long long h_hist[kHistWords] = {0};
    cudaError_t e = dev_alloc((void **)&d_hist, sizeof(h_hist));
    if (e == cudaSuccess) e = cudaMemsetAsync(d_hist, 0, sizeof(h_hist), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->err + kErrBadCol, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) {
        const int64_t blocks = std::min<int64_t>((p->M + 7) / 8, (int64_t)p->num_sms * 8);
        k_check_cols<<<(unsigned)std::max<int64_t>(1, blocks), 256, 0, s>>>(
            p->rowptr, col, p->M, p->K, p->row0, p->t_split, p->chunk, p->chunks, p->n_chunks,
            p->err, d_hist);
        count_launch();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(&flag, p->err + kErrBadCol, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h_hist, d_hist, sizeof(h_hist), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    dev_free(d_hist);
    if (e != cudaSuccess) return from_cuda(e);
    if (flag) return SPMM_ERR_INVALID_INPUT;
    // window half-width: the smallest 2^b (b <= 12) holding >= 85% of the entries
    unsigned long long total = 0, cum = 0;
    for (int b = 0; b < kSpreadBins; ++b) {
        p->spread_hist[b] = (int64_t)h_hist[b];
        total += h_hist[b];
    }
    p->spread_known = true;
    p->blk_intra = (int64_t)h_hist[kSpreadBins];
    p->rows_sorted = h_hist[kSpreadBins + 1] == 0;
    p->band_w = 0;
    p->band_cover = 0.0;
    for (int b = 0; b <= 12 && total > 0; ++b) {
        cum += h_hist[b];
        const double cover = (double)cum / (double)total;
        if (b >= 1 && cover >= 0.85) {
            p->band_w = (int64_t)1 << b;
            p->band_cover = cover;
            p->band_all = (cum == total);
            break;
        }
    }
    return SPMM_OK;
}

spmm_status spmm_plan_prepare_blocks(spmm_plan_t plan, const int32_t *col, const float *val,
                                     void *stream) {
    if (!plan) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    if (p->nnz > 0 && !col) return SPMM_ERR_INVALID_ARG;
    if (p->row0 != 0) return SPMM_ERR_UNSUPPORTED;
    if (col) col += p->col_base;
    if (val) val += p->col_base;
    return from_cuda(block_prepare(p, col, val, (cudaStream_t)stream));
}

spmm_status spmm_plan_sync(spmm_plan_t plan, void *stream) {
    if (!plan) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    cudaStream_t s = (cudaStream_t)stream;
    int32_t words[kErrWords] = {0};
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(words, p->err, sizeof(words), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p->err, 0, sizeof(words));
    if (e != cudaSuccess) return from_cuda(e);
    if (words[kErrTimeout]) return SPMM_ERR_TIMEOUT;
    return SPMM_OK;
}

spmm_status spmm_run(spmm_plan_t plan, const int32_t *col, const float *val, const float *B,
                     int64_t N, spmm_reduce reduce, float *C, int32_t *argmax, void *stream) {
    return spmm_run_ex(plan, col, val, B, N, reduce, nullptr, SPMM_ACT_NONE, C, argmax, stream);
}

spmm_status spmm_run_ex(spmm_plan_t plan, const int32_t *col, const float *val, const float *B,
                        int64_t N, spmm_reduce reduce, const float *bias, spmm_activation act,
                        float *C, int32_t *argmax, void *stream) {
    if (!plan || N < 0 || reduce < SPMM_SUM || reduce > SPMM_MAX) return SPMM_ERR_INVALID_ARG;
    if (act != SPMM_ACT_NONE && act != SPMM_ACT_RELU) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    if (p->M == 0 || N == 0) return SPMM_OK;
    if (!C) return SPMM_ERR_INVALID_ARG;
    if (p->nnz > 0 && (!col || !B)) return SPMM_ERR_INVALID_ARG;
    if (N >= INT32_MAX / 4) return SPMM_ERR_UNSUPPORTED;
    if (reduce != SPMM_MAX) argmax = nullptr;
    // a row-range plan reads its rows' entries out of the full arrays
    if (col) col += p->col_base;
    if (val) val += p->col_base;
    const int aligned = (((uintptr_t)B % 16 == 0) && ((uintptr_t)C % 16 == 0) &&
                         ((uintptr_t)argmax % 16 == 0) ? 1 : 0) |
                        (((uintptr_t)col % 16 == 0) && ((uintptr_t)val % 16 == 0) ? 2 : 0) |
                        (val == nullptr ? 4 : 0);
    spmm_plan_info r;
    fill_desc(p, &r);
    route_fill(&r, N, reduce, aligned, p->num_sms, p->family_override, &r);
    if (r.col_tiles > kMaxTilesY) return SPMM_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;

    RunArgs a{};
    a.rowptr = p->rowptr;
    a.col = col;
    a.val = val;
    a.B = B;
    a.C = C;
    a.argmax = argmax;
    a.M = p->M;
    a.K = p->K;
    a.nnz4 = (int32_t)(p->nnz & ~(int64_t)3);
    a.N = (int32_t)N;
    a.n_vec = (int32_t)((N + r.vec - 1) / r.vec);
    a.t_split = (int32_t)p->t_split;
    a.chunk = (int32_t)p->chunk;
    a.n_chunks = (int32_t)p->n_chunks;
    a.n_heavy = (int32_t)p->n_heavy;
    a.chunks = p->chunks;
    a.heavy_rows = p->heavy_rows;
    a.heavy_chunk0 = p->heavy_chunk0;
    a.err = p->err;
    a.bias = bias;
    a.act = (int32_t)act;
    a.rows_sorted = p->rows_sorted ? 1 : 0;
    a.row0 = p->row0;
    a.seg_tiles = p->seg_tiles;
    a.seg_n_tiles = p->seg_n_tiles;
    if (r.family == SPMM_FAMILY_STREAM) {
        // the per-entry row ids are built once per plan, on its first run
        if (!p->ga_rid) {
            cudaError_t e = gather_prepare(p, s);
            if (e != cudaSuccess) return from_cuda(e);
        }
        spmm_status st = ensure_workspace(p, (size_t)r.workspace_bytes);
        if (st != SPMM_OK) return st;
        a.ga_rid = p->ga_rid;
        char *wb = reinterpret_cast<char *>(p->work);
        const size_t meta = ((size_t)r.stream_ranges * sizeof(int4) + 255) / 256 * 256;
        const size_t vals = (size_t)r.col_tiles * (size_t)r.stream_ranges * 2 * 4 *
                            (size_t)r.lanes * 4;
        a.seg_meta = reinterpret_cast<int4 *>(wb);
        a.seg_cval = reinterpret_cast<float *>(wb + meta);
        a.seg_carg = reduce == SPMM_MAX ? reinterpret_cast<int32_t *>(wb + meta + vals) : nullptr;
        return from_cuda(launch_stream(a, reduce, val != nullptr, r.lanes, r.stream_ranges,
                                       r.col_tiles, s));
    }
    if (r.family == SPMM_FAMILY_GATHER) {
        // the per-entry row ids are built once per plan, on the first GATHER run
        if (!p->ga_rid) {
            cudaError_t e = gather_prepare(p, s);
            if (e != cudaSuccess) return from_cuda(e);
        }
        spmm_status st = ensure_workspace(p, (size_t)r.workspace_bytes);
        if (st != SPMM_OK) return st;
        a.ga_rid = p->ga_rid;
        char *wb = reinterpret_cast<char *>(p->work);
        const size_t meta = ((size_t)r.gather_ctas * sizeof(int4) + 255) / 256 * 256;
        const size_t vals = (size_t)r.col_tiles * (size_t)r.gather_ctas * 2 *
                            (size_t)gather_tile(N) * 4;
        a.seg_meta = reinterpret_cast<int4 *>(wb);
        a.seg_cval = reinterpret_cast<float *>(wb + meta);
        a.seg_carg = reduce == SPMM_MAX ? reinterpret_cast<int32_t *>(wb + meta + vals) : nullptr;
        return from_cuda(launch_gather(a, reduce, val != nullptr, r.gather_ctas, r.col_tiles, s));
    }
    if (r.family == SPMM_FAMILY_SEGMENT) {
        spmm_status st = ensure_workspace(p, (size_t)r.workspace_bytes);
        if (st != SPMM_OK) return st;
        a.seg_warps = r.seg_warps;
        char *wb = reinterpret_cast<char *>(p->work);
        const size_t meta = ((size_t)r.seg_warps * sizeof(int4) + 255) / 256 * 256;
        const size_t vals = (size_t)r.col_tiles * (size_t)r.seg_warps * 2 *
                            (4 * (size_t)r.lanes * (size_t)r.seg_chunks) * 4;
        a.seg_meta = reinterpret_cast<int4 *>(wb);
        a.seg_cval = reinterpret_cast<float *>(wb + meta);
        a.seg_carg = reduce == SPMM_MAX ? reinterpret_cast<int32_t *>(wb + meta + vals) : nullptr;
        return from_cuda(launch_segment(a, r.lanes, r.seg_chunks, reduce, val != nullptr,
                                        r.col_tiles, s));
    }
    const bool split = p->n_heavy > 0 && r.family != SPMM_FAMILY_BLOCK;
    if (split) {
        spmm_status st = ensure_workspace(p, workspace_need(p, N, reduce));
        if (st != SPMM_OK) return st;
        a.ws_val = reinterpret_cast<float *>(p->work);
        a.ws_arg = reduce == SPMM_MAX
                       ? reinterpret_cast<int32_t *>(reinterpret_cast<char *>(p->work) +
                                                     (size_t)p->n_chunks * (size_t)N * 4)
                       : nullptr;
    }
    const bool has_val = val != nullptr;
    cudaError_t e;
    if (r.family == SPMM_FAMILY_BLOCK) {
        // A's diagonal blocks are prepared once per plan and flavour of A
        if (p->bk_flavor != (has_val ? 1 : 0)) {
            e = block_prepare(p, col, val, s);
            if (e != cudaSuccess) return from_cuda(e);
        }
        spmm_status st = ensure_workspace(p, (size_t)r.workspace_bytes);
        if (st != SPMM_OK) return st;
        a.bk_p = reinterpret_cast<float *>(p->work);
        a.bk_a = p->bk_tiles;
        a.bk_off_rowptr = p->bk_off_rowptr;
        a.bk_off_col = p->bk_off_col;
        a.bk_off_val = p->bk_off_val;
        e = launch_block(a, reduce, has_val, s);
    } else if (r.family == SPMM_FAMILY_WINDOW) {
        WinShape w;
        const int rpg = (int)((int64_t)r.window_rows * r.lanes / (kWarp * 16));
        window_shape(p->M, p->K, N, p->dbar, p->band_w, has_val, r.lanes, r.window_chunks, rpg,
                     &w);
        e = launch_window(a, w, reduce, has_val, !p->band_all, r.window_ctas,
                          r.col_tiles, s);
    } else if (r.family == SPMM_FAMILY_COLTILE) {
        // warps per row: the column tiles, up to a CTA's 8 warps (a power of two)
        int wpr = 1;
        while (wpr < r.col_tiles && wpr < 8) wpr <<= 1;
        const int tiles_y = (r.col_tiles + wpr - 1) / wpr;
        if (tiles_y > kMaxTilesY) return SPMM_ERR_UNSUPPORTED;
        e = launch_coltile(a, wpr, tiles_y, reduce, has_val, (aligned & 2) != 0, s);
    } else if (r.family == SPMM_FAMILY_ROWGROUP)
        e = launch_rowgroup(a, r.vec, r.lanes, reduce, has_val, r.col_tiles, s);
    else
        e = launch_warprow(a, r.vec, r.lanes, reduce, has_val, r.col_tiles, s);
    if (e == cudaSuccess && split) {
        // the split rows take the lane shape of the row-per-warp families (the
        // WINDOW family's lanes cover only part of its column tile)
        int64_t hl = r.lanes, ht = r.col_tiles;
        if (r.family == SPMM_FAMILY_WINDOW) {
            hl = std::min<int64_t>(32, std::max<int64_t>(2, pow2ceil(a.n_vec)));
            ht = (a.n_vec + hl - 1) / hl;
        }
        e = launch_heavy(a, r.vec, (int)hl, reduce, has_val, (int)ht, s);
    }
    return from_cuda(e);
}

}  // extern "C"
