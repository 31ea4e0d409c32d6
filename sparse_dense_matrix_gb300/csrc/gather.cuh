// GATHER family: the B rows of a skewed graph at wide N are fetched by the
// tensor-copy engine (TMA `tile::gather4`, four rows per instruction) into a
// shared-memory ring, instead of by the threads that reduce them.
//
// The stored entries are cut into equal contiguous ranges, one per CTA
// (entry-balanced: a hub row of 1e5 entries spreads over several CTAs, and no
// row waits on another; ParamSpMM section 3.2, nonzero-split workload
// balancing). Each CTA has one producer warp and four consumer warps:
//   * the producer streams its range's columns, values and row ids (the
//     plan's per-entry row array) eight stages ahead of use, writes each
//     stage's E entries into a small header, and issues E / 4 gather4 copies
//     of the entries' B rows (the CTA's column tile of CT columns) into the
//     stage, completing on the stage's mbarrier;
//   * the consumer warps own CT / 4 columns each and walk every entry of the
//     stage in CSR order, so each keeps its running row in registers with no
//     exchange between warps: a row is finished (mean, epilogue, store) when
//     the next entry's row id differs, and the rows with no entry in between
//     are written as empty rows.
// The dependent rowptr -> col -> B chain of a row-per-warp kernel becomes a
// stream: the column ids are loaded long before their rows are needed, and
// the rows in flight are bounded by the ring (96 KB per CTA, two CTAs per
// SM), not by registers (graph-spmm card, "Requirements and limits": hubs
// want a segmented schedule; DualGCN section 3.3: independent gathers in
// flight). The rows open at the two ends of a CTA's range leave as partials
// that k_segment_fix combines in CTA order, as for the SEGMENT family; every
// summation order is fixed by the plan, N and the grid (bitwise
// reproducible, no atomics).
#pragma once

#include "common.cuh"
#include "segment.cuh"
#include "tma.cuh"

namespace spmm {

#ifndef SPMM_GA_STAGES
#define SPMM_GA_STAGES 6
#endif
constexpr int kGaStages = SPMM_GA_STAGES;
constexpr int kGaStageFloats = 4096;      // 16 KB of gathered B rows per stage
constexpr int kGaConsumers = 4;           // consumer warps; the producer is warp 4
constexpr int kGaThreads = (kGaConsumers + 1) * kWarp;
constexpr int kGaAhead = 8;               // stages whose entries the producer holds in registers
constexpr int kGaMaxE = 32;               // entries per stage: one per producer lane at most

struct GaHeader {                          // one stage's entries, written by the producer
    int rid[kGaMaxE];
    float val[kGaMaxE];
    int col[kGaMaxE];
};
constexpr int kGaRingBytes = kGaStages * kGaStageFloats * 4;
constexpr int kGaSmemBytes =
    128 + kGaRingBytes + kGaStages * (int)sizeof(GaHeader) + 2 * kGaStages * 8;
static_assert(sizeof(GaHeader) % 16 == 0, "16-byte header rows");

template <int V>
__device__ __forceinline__ void ga_lds(const float *p, float (&x)[V]) {
    if constexpr (V == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        x[0] = *p;
    }
}
template <int V>
__device__ __forceinline__ void ga_st(float *p, const float (&x)[V]) {
    if constexpr (V == 2) __stcs(reinterpret_cast<float2 *>(p), make_float2(x[0], x[1]));
    else __stcs(p, x[0]);
}
template <int V>
__device__ __forceinline__ void ga_st_i(int32_t *p, const int (&x)[V]) {
    if constexpr (V == 2) __stcs(reinterpret_cast<int2 *>(p), make_int2(x[0], x[1]));
    else __stcs(p, x[0]);
}

// CT: columns of the CTA's tile (128 or 256); E = 4096 / CT entries per stage;
// every consumer lane owns V = CT / 128 adjacent columns.
template <int CT, int RED, bool HAS_VAL, bool EPI>
__global__ void __launch_bounds__(kGaThreads, 2) k_gather(const RunArgs a,
                                                       const __grid_constant__ CUtensorMap bmap) {
    constexpr int E = kGaStageFloats / CT;
    constexpr int V = CT / (kWarp * kGaConsumers);
    static_assert(E >= 4 && E <= kGaMaxE && E % 4 == 0 && (V == 1 || V == 2), "stage shape");
    constexpr unsigned FULL = 0xffffffffu;
    using A = Acc<V, RED, HAS_VAL>;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    float *ring = reinterpret_cast<float *>(smem);
    GaHeader *hdr = reinterpret_cast<GaHeader *>(smem + kGaRingBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kGaRingBytes +
                                                  kGaStages * sizeof(GaHeader));
    uint64_t *empty = full + kGaStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & (kWarp - 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGaStages; ++s) {
            mbar_init(&full[s], kWarp);          // every producer lane arrives
            mbar_init(&empty[s], kGaConsumers);  // one arrival per consumer warp
        }
        mbar_init_fence();
    }
    __syncthreads();

    // this CTA's entries [e0, e1); the host launches at most nnz CTAs, so the
    // range is never empty
    const int64_t nnz = a.rowptr[a.M];
    const int W = gridDim.x, k = blockIdx.x;
    const int64_t e0 = nnz * k / W, e1 = nnz * (k + 1) / W;
    const int T = (int)((e1 - e0 + E - 1) / E);

    if (warp == kGaConsumers) {
        // ---- producer
        int pc[kGaAhead], pr[kGaAhead];
        float pv[kGaAhead];
        auto fetch = [&](int t, int d) {
            const int64_t p = e0 + (int64_t)t * E + lane;
            const bool in = lane < E && t < T && p < e1;
            // padding entries gather B row 0 and carry no row
            pc[d] = in ? ld_stream(a.col + p) : 0;
            pr[d] = in ? ld_stream(a.ga_rid + p) : -1;
            pv[d] = (HAS_VAL && in) ? ld_stream(a.val + p) : 1.0f;
        };
#pragma unroll
        for (int d = 0; d < kGaAhead; ++d) fetch(d, d);
        int issued = 0;
        bool ok = true;
        for (int t0 = 0; t0 < T && ok; t0 += kGaAhead) {
#pragma unroll
            for (int d = 0; d < kGaAhead; ++d) {
                const int t = t0 + d;
                if (t >= T) break;
                const int s = t % kGaStages;
                if (t >= kGaStages) {
                    const bool w = mbar_wait(&empty[s], (uint32_t)(t / kGaStages - 1) & 1u, a.err);
                    if (!__all_sync(FULL, w)) {
                        ok = false;
                        break;
                    }
                }
                const int c = pc[d], r = pr[d];
                const float v = pv[d];
                fetch(t + kGaAhead, d);
                if (lane < E) {
                    hdr[s].rid[lane] = r;
                    hdr[s].val[lane] = v;
                    hdr[s].col[lane] = c;
                }
                const int q = (lane * 4) & (kWarp - 1);
                const int c0 = __shfl_sync(FULL, c, q), c1 = __shfl_sync(FULL, c, q + 1);
                const int c2 = __shfl_sync(FULL, c, q + 2), c3 = __shfl_sync(FULL, c, q + 3);
                // each lane's arrival releases its header stores to the consumers
                if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(E * CT * 4));
                else mbar_arrive(&full[s]);
                if (lane < E / 4)
                    gather4_g2s(ring + (size_t)s * kGaStageFloats + (size_t)lane * 4 * CT, &bmap,
                                (int)blockIdx.y * CT, c0, c1, c2, c3, &full[s]);
                issued = t + 1;
            }
        }
        if (!ok) {
            // never leave while copies this warp issued may still be landing
            for (int t = max(0, issued - kGaStages); t < issued; ++t)
                mbar_wait(&full[t % kGaStages], (uint32_t)(t / kGaStages) & 1u, a.err);
        }
        return;
    }

    // ---- consumers: warp `warp` owns columns cl .. cl + V - 1 of every row
    const int64_t N = a.N;
    const int coff = warp * kWarp * V + lane * V;    // offset inside the column tile
    const int64_t cl = (int64_t)blockIdx.y * CT + coff;
    const int first_row = a.ga_rid[e0], last_row = a.ga_rid[e1 - 1];
    const bool head_open = e0 > 0 && a.ga_rid[e0 - 1] == first_row;
    const bool tail_open = e1 < nnz && a.ga_rid[e1] == last_row;
    const int64_t next_row = e1 < nnz ? (int64_t)a.ga_rid[e1] : a.M;

    auto store_row = [&](int64_t row, const A &x, int d) {
        float out[V];
        int arg[V];
        x.finish(d, out, arg);
        if constexpr (RED == SPMM_SUM) mean_scale<V>(a, d, out);
        if constexpr (EPI) epilogue<V>(a, cl, out);
        ga_st<V>(a.C + row * N + cl, out);
        if (RED == SPMM_MAX && a.argmax) ga_st_i<V>(a.argmax + row * N + cl, arg);
    };
    auto empty_rows = [&](int64_t r0, int64_t r1) {  // rows [r0, r1) hold no entry
        A z;
        z.init();
        for (int64_t r = r0; r < r1; ++r) store_row(r, z, 0);
    };
    // an open row's partial: slot 0 the row open at the start of the range,
    // slot 1 the row open at its end (the layout k_segment_fix reads)
    auto store_carry = [&](int slot, const A &x) {
        const int64_t o = (((int64_t)blockIdx.y * W + k) * 2 + slot) * CT + coff;
        ga_st<V>(a.seg_cval + o, x.v);
        if constexpr (RED == SPMM_MAX) ga_st_i<V>(a.seg_carg + o, x.j);
    };

    if (e0 == 0) empty_rows(0, first_row);
    A acc;
    acc.init();
    int cur = first_row, cnt = 0, h0_ends = 0, tail_row = -1;
    bool head = head_open, failed = false;
    for (int t = 0; t < T; ++t) {
        const int s = t % kGaStages;
        const bool w = mbar_wait(&full[s], (uint32_t)(t / kGaStages) & 1u, a.err);
        if (!__all_sync(FULL, w)) {
            failed = true;
            break;
        }
        const GaHeader &h = hdr[s];
        const float *st = ring + (size_t)s * kGaStageFloats + coff;
        const int64_t left = e1 - e0 - (int64_t)t * E;
        const int ne = left < E ? (int)left : E;
        for (int i0 = 0; i0 < ne; i0 += 4) {
            const int4 r4 = *reinterpret_cast<const int4 *>(&h.rid[i0]);
            const int4 c4 = *reinterpret_cast<const int4 *>(&h.col[i0]);
            const float4 v4 = *reinterpret_cast<const float4 *>(&h.val[i0]);
            const int rr[4] = {r4.x, r4.y, r4.z, r4.w};
            const int cc[4] = {c4.x, c4.y, c4.z, c4.w};
            const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float b[4][V];
#pragma unroll
            for (int u = 0; u < 4; ++u) ga_lds<V>(st + (i0 + u) * CT, b[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u >= ne) break;
                if (rr[u] != cur) {                   // row `cur` ended at the previous entry
                    if (head) {
                        store_carry(0, acc);
                        h0_ends = 1;
                        head = false;
                    } else {
                        store_row(cur, acc, cnt);
                    }
                    empty_rows((int64_t)cur + 1, rr[u]);
                    cur = rr[u];
                    cnt = 0;
                    acc.init();
                }
                acc.add(vv[u], cc[u], b[u]);
                ++cnt;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (failed) return;
    if (tail_open) {                                 // the last row goes on past e1
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
    if (warp == 0 && lane == 0 && blockIdx.y == 0)
        a.seg_meta[k] = make_int4(head_open ? first_row : -1, h0_ends, tail_row, 0);
}

namespace gather_detail {
template <int CT, int RED, bool HAS_VAL>
cudaError_t go(const RunArgs &a, const CUtensorMap &map, int ctas, int tiles_y, cudaStream_t s) {
    const bool epi = a.bias != nullptr || a.act != SPMM_ACT_NONE;
    auto kern = epi ? k_gather<CT, RED, HAS_VAL, true> : k_gather<CT, RED, HAS_VAL, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGaSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)ctas, (unsigned)tiles_y), kGaThreads, kGaSmemBytes, s>>>(a, map);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = (int64_t)ctas * (a.N / 4);
    k_segment_fix<RED><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a, CT);
    count_launch();
    return cudaGetLastError();
}
}  // namespace gather_detail

// Launch for one reduction (instantiated per reduction in f_gather_{sum,max}.cu).
// a.seg_warps holds the CTA count of the ranges, a.seg_meta / seg_cval /
// seg_carg the open-row workspace.
template <int RED>
cudaError_t launch_gather_red(const RunArgs &a, const CUtensorMap &map, int ct, bool has_val,
                              int ctas, int tiles_y, cudaStream_t s) {
    if (ct == 256)
        return has_val ? gather_detail::go<256, RED, true>(a, map, ctas, tiles_y, s)
                       : gather_detail::go<256, RED, false>(a, map, ctas, tiles_y, s);
    if (ct == 128)
        return has_val ? gather_detail::go<128, RED, true>(a, map, ctas, tiles_y, s)
                       : gather_detail::go<128, RED, false>(a, map, ctas, tiles_y, s);
    return cudaErrorInvalidValue;
}

extern template cudaError_t launch_gather_red<SPMM_SUM>(const RunArgs &, const CUtensorMap &,
                                                        int, bool, int, int, cudaStream_t);
extern template cudaError_t launch_gather_red<SPMM_MAX>(const RunArgs &, const CUtensorMap &,
                                                        int, bool, int, int, cudaStream_t);

}  // namespace spmm
