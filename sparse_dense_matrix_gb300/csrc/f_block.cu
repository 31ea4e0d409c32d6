// BLOCK family: block-diagonal graphs on the tensor cores (RA-SpMM's
// community regime and its blocked tensor-core kernels; the diagonal blocks of
// a community graph are dense enough that a dense product on tcgen05 moves far
// fewer bytes than per-entry gathers).
//
// A CTA of 128 threads owns rows [r0, r0 + 128) and output columns
// [n0, n0 + 128). Its rows lie in one diagonal block of kBlockRows columns,
// [b0, b0 + kBlockRows). For each chunk of 32 of those columns the CTA
// densifies A's entries into a 128 x 32 tile (thread t owns row r0 + t;
// duplicates are added in CSR order), stages B's 32 x 128 slice, and one
// thread issues tcgen05.mma kind::tf32 into a 128 x 128 fp32 accumulator in
// tensor memory. fp32 operands are split as x = hi + lo with hi and lo TF32
// (round to nearest), and each product is hi_a hi_b + hi_a lo_b + lo_a hi_b,
// about 2^-21 relative per term, inside the fp32 SpMM tolerance (an
// unweighted A has lo_a = 0, so two passes). Operand tiles are K-major, no
// swizzle: 8-row x 16-byte core matrices, 128 bytes apart along K and
// 32 * 4 * 8 bytes apart along rows.
// The epilogue reads the accumulator back (thread t = TMEM lane t = row r0+t),
// adds the row's entries outside the diagonal block in CSR order with fp32
// FMA, applies the mean's 1/d and the fused bias/ReLU, and writes C once.
// Sum and mean only (max needs comparisons, not products).
#include <cstring>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tma.cuh"

namespace spmm {

namespace {

constexpr int kBkThreads = 256;              // warps 0-3: A rows (TMEM lanes 0..127); 4-7: B
constexpr int kBkM = 128;                    // rows per CTA (MMA M)
constexpr int kBkN = 128;                    // output columns per CTA (MMA N, TMEM columns)
constexpr int kBkKC = 32;                    // block columns per staged chunk
constexpr int kBkChunks = kBlockRows / kBkKC;
constexpr uint32_t kLBO = 128;               // next core matrix along K, bytes
constexpr uint32_t kSBO = (kBkKC / 4) * 128; // next 8-row group, bytes
constexpr uint32_t kTileA = kBkM * kBkKC * 4;
constexpr uint32_t kTileB = kBkN * kBkKC * 4;
constexpr int kBkStages = 2;                 // B chunks in flight (tensor copies)
constexpr uint32_t kOffStage = 2 * kTileA + 2 * kTileB;
constexpr uint32_t kOffBars = kOffStage + kBkStages * kBkKC * kBkN * 4;
constexpr int kBkSmem = (int)kOffBars + 64 + 1024;
constexpr int kTilePitch = kBkN + 4;         // accumulator rows in shared memory (floats)
static_assert(kBkM * kTilePitch * 4 <= (int)kOffBars, "the accumulator tile reuses the operand tiles");

// byte offset of element (r, k) in a K-major tile of kBkKC columns
__device__ __forceinline__ uint32_t km_off(int r, int k) {
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
__global__ void __launch_bounds__(kBkThreads) k_block(const RunArgs a,
                                                     const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint32_t *a_hi = reinterpret_cast<uint32_t *>(sm);
    uint32_t *a_lo = reinterpret_cast<uint32_t *>(sm + kTileA);
    uint32_t *b_hi = reinterpret_cast<uint32_t *>(sm + 2 * kTileA);
    uint32_t *b_lo = reinterpret_cast<uint32_t *>(sm + 2 * kTileA + kTileB);
    float *stage = reinterpret_cast<float *>(sm + kOffStage);        // [kBkStages][KC][kBkN]
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kOffBars);     // [kBkStages]
    uint64_t *mma_bar = full + kBkStages;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(mma_bar + 1);

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t r0 = (int64_t)blockIdx.x * kBkM;
    const int n0 = blockIdx.y * kBkN;
    const int n_eff = min(kBkN, a.N - n0);                // a multiple of 16
    const int64_t b0 = r0 / kBlockRows * kBlockRows;      // first column of the diagonal block
    const int64_t N = a.N;
    // warps w and w + 4 share TMEM lanes 32 (w % 4) .. +31: the rows of the tile
    const int rl = (warp & 3) * 32 + lane;
    const int64_t row = r0 + rl;
    const bool has_row = row < a.M;
    const int p0 = has_row ? a.rowptr[row] : 0;
    const int p1 = has_row ? a.rowptr[row + 1] : 0;
    const bool a_side = warp < 4;                         // warps 0-3 densify A, 4-7 convert B

    if (t == 0) {
        for (int st = 0; st < kBkStages; ++st) mbar_init(&full[st], 1);
        mbar_init(mma_bar, 1);
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
    const uint32_t id = instr_desc(kBkM, n_eff);
    constexpr int kPasses = HAS_VAL ? 3 : 2;
    constexpr uint32_t kStageBytes = kBkKC * kBkN * 4;

    // B chunks come by 2-D tensor copies (rows past K and columns past N read
    // as zeros), kBkStages ahead of their conversion
    const int tma_thread = 4 * kWarp;
    int issued = 0, converted = 0;        // chunks requested / taken from the staging ring
    if (t == tma_thread) {
        for (int kc = 0; kc < kBkStages && kc < kBkChunks; ++kc, ++issued) {
            mbar_arrive_expect_tx(&full[kc], kStageBytes);
            tensor2d_g2s(stage + (size_t)kc * kBkKC * kBkN, &bmap, n0, (int)(b0 + kc * kBkKC),
                         &full[kc]);
        }
    }

    // Sorted rows: the entries of the block are [qa, qb). They are read through
    // an 8-entry register buffer (jb, wb) refilled by 8 independent loads, and
    // consumed in order (a prefix of the buffer per chunk).
    int q = p0, qa = p0, nb = 0, cons = 0;
    int jb[8];
    float wb[8];
    auto refill = [&]() {
        q += nb;
        nb = min(8, p1 - q);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            jb[u] = u < nb ? __ldg(a.col + q + u) : INT_MAX;
            wb[u] = (HAS_VAL && u < nb) ? __ldg(a.val + q + u) : 1.0f;
        }
        cons = 0;
    };
    if (a_side && a.rows_sorted) {
        while (q < p1 && (int64_t)a.col[q] < b0) ++q;
        qa = q;
        refill();
    }
    bool ok = true;
    for (int kc = 0; kc < kBkChunks && ok; ++kc) {
        const int64_t c0 = b0 + (int64_t)kc * kBkKC;
        const int st = kc % kBkStages;
        if (a_side) {
            // ---- A: this thread's row; fp32 sums staged in the lo tile, then split
            float *tmp = reinterpret_cast<float *>(a_lo);
#pragma unroll
            for (int k4 = 0; k4 < kBkKC / 4; ++k4)
                *reinterpret_cast<float4 *>(tmp + (km_off(rl, 4 * k4) >> 2)) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a.rows_sorted) {
                while (nb > 0) {
                    int used = cons;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (u >= cons && u < nb && (int64_t)jb[u] < c0 + kBkKC) {
                            tmp[km_off(rl, (int)((int64_t)jb[u] - c0)) >> 2] += wb[u];
                            used = u + 1;
                        }
                    }
                    cons = used;
                    if (cons < nb) break;             // the rest belongs to later chunks
                    refill();
                }
            } else {
                for (int p = p0; p < p1; ++p) {
                    const int64_t c = a.col[p];
                    if ((uint64_t)(c - c0) < (uint64_t)kBkKC)
                        tmp[km_off(rl, (int)(c - c0)) >> 2] += HAS_VAL ? a.val[p] : 1.0f;
                }
            }
#pragma unroll
            for (int k4 = 0; k4 < kBkKC / 4; ++k4) {
                const uint32_t o = km_off(rl, 4 * k4) >> 2;
                const float4 v = *reinterpret_cast<const float4 *>(tmp + o);
                uint4 h, l;
                h.x = to_tf32(v.x); l.x = to_tf32(v.x - __uint_as_float(h.x));
                h.y = to_tf32(v.y); l.y = to_tf32(v.y - __uint_as_float(h.y));
                h.z = to_tf32(v.z); l.z = to_tf32(v.z - __uint_as_float(h.z));
                h.w = to_tf32(v.w); l.w = to_tf32(v.w - __uint_as_float(h.w));
                *reinterpret_cast<uint4 *>(a_hi + o) = h;
                *reinterpret_cast<uint4 *>(a_lo + o) = l;
            }
        } else {
            // ---- B: the staged row-major chunk [KC][kBkN] -> the N x K operand
            const bool landed = mbar_wait_poll(&full[st], (uint32_t)(kc / kBkStages) & 1u, a.err);
            if (landed) {
                const float *src = stage + (size_t)st * kBkKC * kBkN;
                const int i = t - 4 * kWarp;                  // 0..127
#pragma unroll 8
                for (int e = i; e < kBkKC * kBkN; e += 4 * kWarp) {
                    const int k = e / kBkN, n = e % kBkN;
                    const float v = src[e];
                    const uint32_t o = km_off(n, k) >> 2;
                    const uint32_t h = to_tf32(v);
                    b_hi[o] = h;
                    b_lo[o] = to_tf32(v - __uint_as_float(h));
                }
            }
            ok = landed;
        }
        // make the tiles visible to the tensor cores, then one thread issues
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        ok = __syncthreads_and(ok);
        if (!ok) break;
        converted = kc + 1;
        if (t == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t A_[2] = {smem_addr(a_hi), smem_addr(a_lo)};
            const uint32_t B_[2] = {smem_addr(b_hi), smem_addr(b_lo)};
            const int pa[3] = {0, 0, 1}, pb[3] = {0, 1, 0};
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps)
#pragma unroll
                for (int ks = 0; ks < kBkKC / 8; ++ks)
                    mma_tf32(tmem, smem_desc(A_[pa[ps]] + (uint32_t)ks * 2u * kLBO),
                             smem_desc(B_[pb[ps]] + (uint32_t)ks * 2u * kLBO), id,
                             (kc | ps | ks) != 0);
            asm volatile(
                "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                    smem_addr(mma_bar))
                : "memory");
        }
        // stage st has been converted: refill it with chunk kc + kBkStages
        if (t == tma_thread && kc + kBkStages < kBkChunks) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&full[st], kStageBytes);
            tensor2d_g2s(stage + (size_t)st * kBkKC * kBkN, &bmap, n0,
                         (int)(b0 + (kc + kBkStages) * kBkKC), &full[st]);
            ++issued;
        }
        // the operand tiles are rewritten by the next chunk: wait for the MMAs
        ok = __syncthreads_and(mbar_wait_poll(mma_bar, (uint32_t)kc & 1u, a.err));
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    // never leave while a tensor copy may still be landing in this CTA's memory
    // (only after an early exit are requested chunks left unconverted)
    if (t == tma_thread)
        for (int kc = converted; kc < issued; ++kc)
            mbar_wait_poll(&full[kc % kBkStages], (uint32_t)(kc / kBkStages) & 1u, a.err);
    const int qb = q + cons;              // first entry past the block (sorted rows, A side)

    if (ok) {
        // The accumulator goes through shared memory (the operand and staging
        // tiles are free now) so that rows can be finished warp-cooperatively:
        // lanes across columns, one coalesced B-row read per entry outside the
        // diagonal block. Per element the order stays: the block's dense sum,
        // then the other entries in CSR order.
        __shared__ int s_qa[kBkM], s_qb[kBkM];
        if (a_side) {
            s_qa[rl] = qa;
            s_qb[rl] = qb;
        }
        float *tile = reinterpret_cast<float *>(sm);       // [kBkM][kTilePitch]
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        for (int c = (warp >> 2) * 16; c < n_eff; c += 32) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c, v);
            float4 *dst = reinterpret_cast<float4 *>(tile + rl * kTilePitch + c);
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4)
                dst[e4] = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
        }
        __syncthreads();
        const int cl = 4 * lane;                            // this lane's 4 columns
        const bool col_ok = cl < n_eff;
        const int cc = col_ok ? cl : 0;
        for (int rr = warp; rr < kBkM; rr += kBkThreads / kWarp) {
            const int64_t i = r0 + rr;
            if (i >= a.M) break;
            const int e0 = a.rowptr[i], e1 = a.rowptr[i + 1];
            float4 acc = *reinterpret_cast<const float4 *>(tile + rr * kTilePitch + cc);
            const float *Bc = a.B + n0 + cc;
            auto add4 = [&](int pb, int pe) {               // entries [pb, pe), 4 in flight
                int p = pb;
                for (; p + 4 <= pe; p += 4) {
                    int j[4];
                    float w[4];
                    float4 x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        j[u] = __ldg(a.col + p + u);
                        w[u] = HAS_VAL ? __ldg(a.val + p + u) : 1.0f;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) x[u] = __ldg(reinterpret_cast<const float4 *>(Bc + (int64_t)j[u] * N));
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc.x = __fmaf_rn(w[u], x[u].x, acc.x);
                        acc.y = __fmaf_rn(w[u], x[u].y, acc.y);
                        acc.z = __fmaf_rn(w[u], x[u].z, acc.z);
                        acc.w = __fmaf_rn(w[u], x[u].w, acc.w);
                    }
                }
                for (; p < pe; ++p) {
                    const int j = __ldg(a.col + p);
                    const float w = HAS_VAL ? __ldg(a.val + p) : 1.0f;
                    const float4 x = __ldg(reinterpret_cast<const float4 *>(Bc + (int64_t)j * N));
                    acc.x = __fmaf_rn(w, x.x, acc.x);
                    acc.y = __fmaf_rn(w, x.y, acc.y);
                    acc.z = __fmaf_rn(w, x.z, acc.z);
                    acc.w = __fmaf_rn(w, x.w, acc.w);
                }
            };
            if (a.rows_sorted) {
                add4(e0, s_qa[rr]);
                add4(s_qb[rr], e1);
            } else {
                for (int p = e0; p < e1; ++p) {
                    const int j = __ldg(a.col + p);
                    if ((uint64_t)((int64_t)j - b0) < (uint64_t)kBlockRows) continue;
                    const float w = HAS_VAL ? __ldg(a.val + p) : 1.0f;
                    const float4 x = __ldg(reinterpret_cast<const float4 *>(Bc + (int64_t)j * N));
                    acc.x = __fmaf_rn(w, x.x, acc.x);
                    acc.y = __fmaf_rn(w, x.y, acc.y);
                    acc.z = __fmaf_rn(w, x.z, acc.z);
                    acc.w = __fmaf_rn(w, x.w, acc.w);
                }
            }
            float out[4] = {acc.x, acc.y, acc.z, acc.w};
            if (RED == SPMM_MEAN) {
                const int d = e1 - e0;
                const float inv_d = d > 0 ? rcp_approx((float)d) : 0.0f;
#pragma unroll
                for (int e = 0; e < 4; ++e) out[e] = __fmul_rn(out[e], inv_d);
            }
            if (col_ok) {
                epilogue<4>(a, (int64_t)n0 + cl, out);
                st_vec<4>(a.C + i * N + n0 + cl, out);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBkN)
                     : "memory");
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
    const unsigned gx = (unsigned)((a.M + kBkM - 1) / kBkM);
    const unsigned gy = (unsigned)((a.N + kBkN - 1) / kBkN);
    kern<<<dim3(gx, gy), kBkThreads, kBkSmem, s>>>(a, map);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

// Requires N % 16 == 0, 16-byte aligned B and C, reduce SUM or MEAN.
cudaError_t launch_block(const RunArgs &a, int reduce, bool has_val, cudaStream_t s) {
    if (reduce == SPMM_SUM) return has_val ? go<SPMM_SUM, true>(a, s) : go<SPMM_SUM, false>(a, s);
    if (reduce == SPMM_MEAN) return has_val ? go<SPMM_MEAN, true>(a, s) : go<SPMM_MEAN, false>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace spmm
