// BLOCK family: block-diagonal graphs on the tensor cores (RA-SpMM's
// community regime and its blocked tensor-core kernels; the diagonal blocks of
// a community graph are dense enough that a dense product on tcgen05 moves far
// fewer bytes than per-entry gathers).
//
// A is fixed, so its share of the work is done once per plan
// (block_prepare): the diagonal block of every 128-row tile (the kBlockRows
// columns [b0, b0 + kBlockRows) that hold its rows' own community) is
// densified (duplicates added in CSR order, fp32) and split as x = hi + lo
// with hi and lo TF32 (round to nearest), stored in the tensor cores' K-major
// operand layout, one 8 KB piece per 16 block columns; the entries outside
// the block are copied into a compact CSR of their own. A launch then only
// streams these pieces:
//   * warp 0 (one thread) bulk-copies the chunk's A pieces (hi, and lo when A
//     is weighted) and loads B's 16 x 128 chunk by a 2-D tensor copy, into a
//     two-stage mbarrier ring;
//   * warps 4-7 split each B chunk into TF32 hi and lo, transposed into the
//     K-major layout;
//   * warp 1 (one thread) issues tcgen05.mma kind::tf32 into a 128 x 128 fp32
//     accumulator in tensor memory: a_hi b_hi + a_hi b_lo + a_lo b_hi (about
//     2^-21 relative per term; two passes for an unweighted A, whose lo is 0)
//     and commits each chunk to the stage's "free" barrier.
// The three roles overlap across the two stages. Meanwhile warps 8-15 take
// the rows' entries outside the diagonal block (lanes across the tile's
// columns, fp32 FMA in CSR order from zero) and write each row's partial to
// the workspace P. The epilogue reads the accumulator back through shared
// memory and finishes the rows warp-cooperatively: block sum + P, the mean's
// 1/d, the fused bias/ReLU, one store of C. Sum and mean only (max needs
// comparisons, not products). Operand tiles are K-major without
// swizzle: 8-row x 16-byte core matrices, 128 bytes apart along K and
// (KC / 4) * 128 bytes apart along rows.
#include <cstring>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tma.cuh"

namespace spmm {

namespace {

constexpr int kBkThreads = 512;              // warps 0-7: the product; 8-15: off-block rows
constexpr int kBkMainWarps = 8;
constexpr int kBkM = 128;                    // rows per CTA (MMA M)
constexpr int kBkN = 128;                    // output columns per CTA (MMA N, TMEM columns)
constexpr int kBkKC = 16;                    // block columns per chunk
constexpr int kBkChunks = kBlockRows / kBkKC;
constexpr uint32_t kLBO = 128;               // next core matrix along K, bytes
constexpr uint32_t kSBO = (kBkKC / 4) * 128; // next 8-row group, bytes
constexpr uint32_t kPiece = kBkM * kBkKC * 4;       // one A piece (8 KB)
constexpr uint32_t kBTile = kBkN * kBkKC * 4;       // one B operand tile (8 KB)
constexpr int kBkStages = 2;
// per stage: A hi, A lo, B as loaded, B hi, B lo
constexpr uint32_t kStageBytes = 2 * kPiece + 3 * kBTile;
constexpr uint32_t kOffBars = kBkStages * kStageBytes;
constexpr int kBkSmem = (int)kOffBars + 128 + 1024;
constexpr int kTilePitch = kBkN + 4;         // accumulator rows in shared memory (floats)
constexpr int kConvThreads = 4 * kWarp;      // warps 4-7
static_assert(kBkM * kTilePitch * 4 <= (int)kOffBars, "the accumulator tile reuses the stages");

// prepared A: [row tile][chunk][hi, lo][kPiece bytes]
constexpr size_t kTileBytes = (size_t)kBkChunks * 2 * kPiece;

// byte offset of element (r, k) in a K-major tile of kBkKC columns
__host__ __device__ __forceinline__ uint32_t km_off(int r, int k) {
    return (uint32_t)(r >> 3) * kSBO + (uint32_t)(k >> 2) * kLBO + (uint32_t)(r & 7) * 16u +
           (uint32_t)(k & 3) * 4u;
}

// shared-memory matrix descriptor: start address, leading (K) and stride
// (row-group) byte offsets in 16-byte units, descriptor version 1, no swizzle
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((kLBO >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((kSBO >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, N >> 3 and M >> 4
__device__ __forceinline__ uint32_t instr_desc(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem, uint64_t a, uint64_t b, uint32_t id,
                                         int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}

template <int RED, bool HAS_VAL>
__global__ void __launch_bounds__(kBkThreads, 2) k_block(const RunArgs a,
                                                     const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kOffBars);   // [stage] A + B landed
    uint64_t *conv = full + kBkStages;                               // [stage] B split
    uint64_t *done = conv + kBkStages;                               // [stage] MMAs read it
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + kBkStages);
    auto stage = [&](int s) { return sm + (size_t)s * kStageBytes; };

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int n0 = blockIdx.x * kBkN;                     // column tiles vary fastest:
    const int64_t tile = blockIdx.y;                      // they share the A pieces in L2
    const int64_t r0 = tile * kBkM;
    const int n_eff = min(kBkN, a.N - n0);                // a multiple of 16
    const int64_t b0 = r0 / kBlockRows * kBlockRows;      // first column of the diagonal block
    const int64_t N = a.N;
    const unsigned char *apiece = reinterpret_cast<const unsigned char *>(a.bk_a) +
                                  (size_t)tile * kTileBytes;

    if (t == 0) {
        for (int s = 0; s < kBkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&conv[s], kConvThreads / kWarp);
            mbar_init(&done[s], 1);
        }
        mbar_init_fence();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tslot)),
                     "r"(kBkN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;
    constexpr int kPasses = HAS_VAL ? 3 : 2;
    constexpr uint32_t kLoadBytes = (HAS_VAL ? 2 : 1) * kPiece + kBTile;

    bool ok = true;
    int issued = 0;                                       // chunks the producer requested
    if (t == 0) {
        // ---------------------------------------------------------- producer
        for (int c = 0; c < kBkChunks && ok; ++c) {
            const int s = c % kBkStages, use = c / kBkStages;
            if (use > 0) ok = mbar_wait_poll(&done[s], (uint32_t)(use - 1) & 1u, a.err);
            if (!ok) break;
            unsigned char *st = stage(s);
            mbar_arrive_expect_tx(&full[s], kLoadBytes);
            bulk_g2s(st, apiece + (size_t)c * 2 * kPiece, kPiece, &full[s]);
            if (HAS_VAL) bulk_g2s(st + kPiece, apiece + (size_t)c * 2 * kPiece + kPiece, kPiece, &full[s]);
            tensor2d_g2s(st + 2 * kPiece, &bmap, n0, (int)(b0 + c * kBkKC), &full[s]);
            issued = c + 1;
        }
    } else if (t == kWarp) {
        // ------------------------------------------------------- MMA issuer
        const uint32_t id = instr_desc(kBkM, n_eff);
        for (int c = 0; c < kBkChunks && ok; ++c) {
            const int s = c % kBkStages, use = c / kBkStages;
            ok = mbar_wait_poll(&conv[s], (uint32_t)use & 1u, a.err);
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t sa = smem_addr(stage(s));
            const uint32_t A_[2] = {sa, sa + kPiece};
            const uint32_t B_[2] = {sa + 2 * kPiece + kBTile, sa + 2 * kPiece + 2 * kBTile};
            const int pa[3] = {0, 0, 1}, pb[3] = {0, 1, 0};
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps)
#pragma unroll
                for (int ks = 0; ks < kBkKC / 8; ++ks)
                    mma_tf32(tmem, smem_desc(A_[pa[ps]] + (uint32_t)ks * 2u * kLBO),
                             smem_desc(B_[pb[ps]] + (uint32_t)ks * 2u * kLBO), id,
                             (c | ps | ks) != 0);
            asm volatile(
                "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                    smem_addr(&done[s]))
                : "memory");
        }
    } else if (warp >= kBkMainWarps) {
        // ------------------------------------------- rows' off-block entries
        // Meanwhile the other eight warps take the rows' entries outside the
        // diagonal block (lanes across the tile's columns, two rows at a time,
        // up to three entries of each per step: six gathers in flight per
        // lane), sum them in CSR order from zero and write the partial row to
        // the workspace P, which the epilogue adds to the block's sum.
        const int cl = 4 * lane;
        const bool col_ok = cl < n_eff;
        const float *Bc = a.B + n0 + (col_ok ? cl : 0);
        const int nrows = (int)(a.M - r0 < kBkM ? a.M - r0 : kBkM);
        constexpr int kWW = kBkThreads / kWarp - kBkMainWarps;   // worker warps
        constexpr int kRB = 2, kEB = 3;
        for (int rr0 = warp - kBkMainWarps; rr0 < nrows; rr0 += kRB * kWW) {
            int qa[kRB], qb[kRB];
            float4 acc[kRB];
#pragma unroll
            for (int k = 0; k < kRB; ++k) {
                const int rr = rr0 + k * kWW;
                const bool live = rr < nrows;
                qa[k] = live ? a.bk_off_rowptr[r0 + rr] : 0;
                qb[k] = live ? a.bk_off_rowptr[r0 + rr + 1] : 0;
                acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            bool more = qa[0] < qb[0] || qa[1] < qb[1];
            while (more) {                                  // uniform across the warp
                int j[kRB][kEB];
                float w[kRB][kEB];
                float4 x[kRB][kEB];
#pragma unroll
                for (int k = 0; k < kRB; ++k)
#pragma unroll
                    for (int u = 0; u < kEB; ++u) {
                        const bool in = qa[k] + u < qb[k];
                        j[k][u] = in ? __ldg(a.bk_off_col + qa[k] + u) : 0;
                        w[k][u] = (HAS_VAL && in) ? __ldg(a.bk_off_val + qa[k] + u) : 1.0f;
                    }
#pragma unroll
                for (int k = 0; k < kRB; ++k)
#pragma unroll
                    for (int u = 0; u < kEB; ++u)
                        if (qa[k] + u < qb[k])
                            x[k][u] = __ldg(reinterpret_cast<const float4 *>(Bc + (int64_t)j[k][u] * N));
                more = false;
#pragma unroll
                for (int k = 0; k < kRB; ++k) {
#pragma unroll
                    for (int u = 0; u < kEB; ++u)
                        if (qa[k] + u < qb[k]) {
                            acc[k].x = __fmaf_rn(w[k][u], x[k][u].x, acc[k].x);
                            acc[k].y = __fmaf_rn(w[k][u], x[k][u].y, acc[k].y);
                            acc[k].z = __fmaf_rn(w[k][u], x[k][u].z, acc[k].z);
                            acc[k].w = __fmaf_rn(w[k][u], x[k][u].w, acc[k].w);
                        }
                    qa[k] += kEB;
                    more |= qa[k] < qb[k];
                }
            }
#pragma unroll
            for (int k = 0; k < kRB; ++k) {
                const int rr = rr0 + k * kWW;
                if (rr < nrows && col_ok)
                    *reinterpret_cast<float4 *>(a.bk_p + (r0 + rr) * N + n0 + cl) = acc[k];
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- B split
        const int i = t - 4 * kWarp;                      // 0..127
        for (int c = 0; c < kBkChunks && ok; ++c) {
            const int s = c % kBkStages, use = c / kBkStages;
            ok = mbar_wait_poll(&full[s], (uint32_t)use & 1u, a.err);
            if (ok && use > 0) ok = mbar_wait_poll(&done[s], (uint32_t)(use - 1) & 1u, a.err);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            unsigned char *st = stage(s);
            const float *src = reinterpret_cast<const float *>(st + 2 * kPiece);   // [KC][kBkN]
            uint32_t *bh = reinterpret_cast<uint32_t *>(st + 2 * kPiece + kBTile);
            uint32_t *bl = reinterpret_cast<uint32_t *>(st + 2 * kPiece + 2 * kBTile);
            // thread i owns column n = i: four k at a time into one 16-byte
            // word of the K-major tile (a quarter-warp stores 128 contiguous bytes)
#pragma unroll
            for (int k4 = 0; k4 < kBkKC / 4; ++k4) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float v = src[(4 * k4 + kk) * kBkN + i];
                    h[kk] = to_tf32(v);
                    l[kk] = to_tf32(v - __uint_as_float(h[kk]));
                }
                const uint32_t o = km_off(i, 4 * k4) >> 2;
                *reinterpret_cast<uint4 *>(bh + o) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(bl + o) = make_uint4(l[0], l[1], l[2], l[3]);
            }
            // the split tiles are read by the tensor cores (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[s]);
        }
    }
    // the accumulator is complete once the last chunk's MMAs have read their
    // stage (a commit tracks every earlier MMA of the issuing thread)
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait_poll(&done[(kBkChunks - 1) % kBkStages],
                                (uint32_t)((kBkChunks - 1) / kBkStages) & 1u, a.err);
    ok = __syncthreads_and(ok);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (ok) {
        // The accumulator goes through shared memory (the stages are free now)
        // so that rows are finished warp-cooperatively: lanes across columns,
        // one coalesced B-row read per entry outside the diagonal block. Per
        // element the order is the block's dense sum, then the other entries
        // in CSR order.
        float *tile_s = reinterpret_cast<float *>(sm);      // [kBkM][kTilePitch]
        const int rl = (warp & 3) * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        for (int c = (warp >> 2) * 16; c < n_eff; c += 16 * (kBkThreads / kWarp / 4)) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c, v);
            float4 *dst = reinterpret_cast<float4 *>(tile_s + rl * kTilePitch + c);
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4)
                dst[e4] = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
        }
        __syncthreads();
        // each warp finishes rows warp, warp + 16, ...: the block's sum plus
        // the off-block partial P (written by this CTA's worker warps; plain
        // coherent loads, ordered by the barrier above), mean, bias/ReLU
        const int cl = 4 * lane;
        const bool col_ok = cl < n_eff;
        const int cc = col_ok ? cl : 0;
        const int nrows = (int)(a.M - r0 < kBkM ? a.M - r0 : kBkM);
        for (int rr = warp; rr < nrows; rr += kBkThreads / kWarp) {
            const int64_t i = r0 + rr;
            const float4 bsum = *reinterpret_cast<const float4 *>(tile_s + rr * kTilePitch + cc);
            float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (col_ok) pv = *reinterpret_cast<const float4 *>(a.bk_p + i * N + n0 + cl);
            float out[4] = {__fadd_rn(bsum.x, pv.x), __fadd_rn(bsum.y, pv.y),
                            __fadd_rn(bsum.z, pv.z), __fadd_rn(bsum.w, pv.w)};
            if (RED == SPMM_MEAN) {
                const int d = a.rowptr[i + 1] - a.rowptr[i];
                const float inv_d = d > 0 ? rcp_approx((float)d) : 0.0f;
#pragma unroll
                for (int e = 0; e < 4; ++e) out[e] = __fmul_rn(out[e], inv_d);
            }
            if (col_ok) {
                epilogue<4>(a, (int64_t)n0 + cl, out);
                st_vec<4>(a.C + i * N + n0 + cl, out);
            }
        }
    } else if (t == 0) {
        // never leave while a copy this CTA requested may still be landing:
        // wait (bounded) for the last request of each stage
        for (int c = max(0, issued - kBkStages); c < issued; ++c)
            mbar_wait_poll(&full[c % kBkStages], (uint32_t)(c / kBkStages) & 1u, a.err);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBkN)
                     : "memory");
}

// ------------------------------------------------------------- preparation
// Densify: one thread per row adds its entries inside the diagonal block into
// the row tile's hi pieces (fp32, CSR order); the pieces start zeroed.
__global__ void k_bk_densify(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ col,
                             const float *__restrict__ val, int64_t M, int64_t K,
                             unsigned char *__restrict__ tiles) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M) return;
    const int64_t tile = i / kBkM, b0 = i / kBlockRows * kBlockRows;
    const int r = (int)(i % kBkM);
    unsigned char *base = tiles + (size_t)tile * kTileBytes;
    for (int p = rowptr[i]; p < rowptr[i + 1]; ++p) {
        const int64_t c = col[p];
        if (c < b0 || c >= b0 + kBlockRows || c >= K) continue;
        const int k = (int)(c - b0), chunk = k / kBkKC;
        float *hi = reinterpret_cast<float *>(base + (size_t)chunk * 2 * kPiece);
        hi[km_off(r, k % kBkKC) >> 2] += val ? val[p] : 1.0f;
    }
}

// Split every fp32 sum of the hi pieces into TF32 hi and lo (lo = 0 when A is
// unweighted: its sums are small integers, exact in TF32).
__global__ void k_bk_split(unsigned char *__restrict__ tiles, int64_t n_pieces) {
    constexpr int kWords = (int)(kPiece / 4);
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n_pieces * kWords;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t piece = q / kWords, w = q % kWords;
        uint32_t *hi = reinterpret_cast<uint32_t *>(tiles + (size_t)piece * 2 * kPiece);
        uint32_t *lo = hi + kWords;
        const float x = __uint_as_float(hi[w]);
        const uint32_t h = to_tf32(x);
        hi[w] = h;
        lo[w] = to_tf32(x - __uint_as_float(h));
    }
}

// The entries outside the diagonal block: per-row counts, then (at the
// scanned offsets) the entries themselves in CSR order.
__global__ void k_bk_off_count(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ col,
                               int64_t M, int32_t *__restrict__ cnt) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M) return;
    const int64_t b0 = i / kBlockRows * kBlockRows;
    int n = 0;
    for (int p = rowptr[i]; p < rowptr[i + 1]; ++p) {
        const int64_t c = col[p];
        n += (c < b0 || c >= b0 + kBlockRows);
    }
    cnt[i] = n;
}

__global__ void k_bk_off_fill(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ col,
                              const float *__restrict__ val, int64_t M,
                              const int32_t *__restrict__ off_rowptr, int32_t *__restrict__ off_col,
                              float *__restrict__ off_val) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M) return;
    const int64_t b0 = i / kBlockRows * kBlockRows;
    int q = off_rowptr[i];
    for (int p = rowptr[i]; p < rowptr[i + 1]; ++p) {
        const int64_t c = col[p];
        if (c >= b0 && c < b0 + kBlockRows) continue;
        off_col[q] = (int32_t)c;
        if (off_val) off_val[q] = val[p];
        ++q;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// B as a 2-D tensor (N columns, K rows) in boxes of kBkN columns x kBkKC rows
cudaError_t encode_b(const RunArgs &a, CUtensorMap *map) {
    std::memset(map, 0, sizeof(*map));
    if (!g_encode) {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kBkN, (cuuint32_t)kBkKC};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.B), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = encode_b(a, &map);
    if (e != cudaSuccess) return e;
    auto kern = k_block<RED, HAS_VAL>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBkSmem);
    if (e != cudaSuccess) return e;
    const unsigned gx = (unsigned)((a.N + kBkN - 1) / kBkN);
    const unsigned gy = (unsigned)((a.M + kBkM - 1) / kBkM);
    kern<<<dim3(gx, gy), kBkThreads, kBkSmem, s>>>(a, map);
    count_launch();
    return cudaGetLastError();
}

void free_prepared(Plan *p) {
    if (p->bk_tiles) cudaFree(p->bk_tiles);
    if (p->bk_off_rowptr) cudaFree(p->bk_off_rowptr);
    if (p->bk_off_col) cudaFree(p->bk_off_col);
    if (p->bk_off_val) cudaFree(p->bk_off_val);
    p->bk_tiles = nullptr;
    p->bk_off_rowptr = nullptr;
    p->bk_off_col = nullptr;
    p->bk_off_val = nullptr;
    p->bk_flavor = -1;
    p->bk_bytes = 0;
    p->bk_n_off = 0;
}

}  // namespace

void block_free(Plan *p) { free_prepared(p); }

size_t block_prepared_bytes(int64_t M, int64_t n_off, bool has_val) {
    const int64_t tiles = (M + kBkM - 1) / kBkM;
    return (size_t)tiles * kTileBytes + 4 * (size_t)(M + 1) + (has_val ? 8 : 4) * (size_t)n_off;
}

cudaError_t block_prepare(Plan *p, const int32_t *col, const float *val, cudaStream_t s) {
    free_prepared(p);
    const int64_t M = p->M;
    if (M == 0) return cudaSuccess;
    const int64_t tiles = (M + kBkM - 1) / kBkM;
    const size_t tbytes = (size_t)tiles * kTileBytes;
    const unsigned grid = (unsigned)((M + 255) / 256);
    cudaError_t e = cudaMalloc(&p->bk_tiles, tbytes);
    if (e == cudaSuccess) e = cudaMalloc((void **)&p->bk_off_rowptr, sizeof(int32_t) * (M + 1));
    if (e == cudaSuccess) e = cudaMemsetAsync(p->bk_tiles, 0, tbytes, s);
    if (e == cudaSuccess) {
        k_bk_densify<<<grid, 256, 0, s>>>(p->rowptr, col, val, M, p->K,
                                          reinterpret_cast<unsigned char *>(p->bk_tiles));
        k_bk_split<<<(unsigned)std::min<int64_t>(tiles * kBkChunks * 8, 65535), 256, 0, s>>>(
            reinterpret_cast<unsigned char *>(p->bk_tiles), tiles * kBkChunks);
        k_bk_off_count<<<grid, 256, 0, s>>>(p->rowptr, col, M, p->bk_off_rowptr);
        count_launch(3);
        e = cudaGetLastError();
    }
    // exclusive scan of the counts on the host (plan time)
    std::vector<int32_t> cnt((size_t)M + 1, 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(cnt.data(), p->bk_off_rowptr, sizeof(int32_t) * M,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        free_prepared(p);
        return e;
    }
    int64_t run = 0;
    for (int64_t i = 0; i < M; ++i) {
        const int32_t c = cnt[i];
        cnt[i] = (int32_t)run;
        run += c;
    }
    cnt[M] = (int32_t)run;
    p->bk_n_off = run;
    e = cudaMemcpyAsync(p->bk_off_rowptr, cnt.data(), sizeof(int32_t) * (M + 1),
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMalloc((void **)&p->bk_off_col, sizeof(int32_t) * std::max<int64_t>(1, run));
    if (e == cudaSuccess && val)
        e = cudaMalloc((void **)&p->bk_off_val, sizeof(float) * std::max<int64_t>(1, run));
    if (e == cudaSuccess) {
        k_bk_off_fill<<<grid, 256, 0, s>>>(p->rowptr, col, val, M, p->bk_off_rowptr,
                                           p->bk_off_col, p->bk_off_val);
        count_launch();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        free_prepared(p);
        return e;
    }
    p->bk_flavor = val ? 1 : 0;
    p->bk_bytes = (int64_t)block_prepared_bytes(M, run, val != nullptr);
    return cudaSuccess;
}

// Requires N % 16 == 0, 16-byte aligned B and C, reduce SUM or MEAN, and the
// plan's prepared blocks (a.bk_*) for this flavour of A.
cudaError_t launch_block(const RunArgs &a, int reduce, bool has_val, cudaStream_t s) {
    if (reduce == SPMM_SUM) return has_val ? go<SPMM_SUM, true>(a, s) : go<SPMM_SUM, false>(a, s);
    if (reduce == SPMM_MEAN) return has_val ? go<SPMM_MEAN, true>(a, s) : go<SPMM_MEAN, false>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace spmm
