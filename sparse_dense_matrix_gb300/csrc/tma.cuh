// Inline-PTX helpers for shared-memory mbarriers and 1-D bulk asynchronous
// copies (global -> shared, completed on an mbarrier's transaction count),
// written from the PTX ISA. Every wait is bounded: after kSpinLimit polls the
// waiter records kErrTimeout in the plan's error words and gives up, so a
// broken invariant surfaces as SPMM_ERR_TIMEOUT instead of a hung GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace spmm {

// A wait gives up after kWaitLimitNs of wall time (read from %globaltimer
// every 256 polls) or kSpinLimit polls, whichever comes first.
constexpr uint32_t kSpinLimit = 1u << 26;
constexpr uint64_t kWaitLimitNs = 500ull * 1000 * 1000;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// make initialised barriers visible to the async (bulk-copy) proxy
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One poll; a waiting thread may be suspended for up to kSuspendNs (it resumes
// as soon as the phase completes), so waiting warps do not spin on the issue slots.
constexpr uint32_t kSuspendNs = 100000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete; false (and the error word set)
// if it has not within the limits above.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 0 && global_ns() - t0 > limit_ns) break;
    }
    atomicOr(err + kErrTimeout, 1);
    return false;
}

// One poll without a suspend hint (returns after a short, implementation-defined
// time); for waits that are expected to end within microseconds.
__device__ __forceinline__ bool mbar_poll(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// mbar_wait with plain polls, bounded the same way.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t *bar, uint32_t parity, int32_t *err) {
    if (mbar_poll(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (mbar_poll(bar, parity)) return true;
        if ((i & 255) == 0 && global_ns() - t0 > kWaitLimitNs) break;
    }
    atomicOr(err + kErrTimeout, 1);
    return false;
}

// Order this thread's earlier generic-proxy accesses of shared memory before its
// later async-proxy ones (a bulk copy into a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory loads by 32-bit shared-window address (volatile: they stay
// after the mbarrier wait that publishes the data).
__device__ __forceinline__ int lds_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void lds_v4(uint32_t addr, float (&b)[4]) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(b[0]), "=f"(b[1]), "=f"(b[2]), "=f"(b[3])
                 : "r"(addr));
}

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tiled tensor copy (box given by the tensor map) of the tile at element
// coordinates (x, y) into this CTA's shared memory (128-byte aligned), completing
// on `bar`. Rows or columns outside the tensor are filled with zeros.
__device__ __forceinline__ void tensor2d_g2s(void *dst, const CUtensorMap *map, int x, int y,
                                             uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_addr(bar))
        : "memory");
}

// Four rows of a 2-D tensor, each one box row of the tensor map (whose box is
// one row high) from column x, into consecutive box rows of this CTA's shared
// memory (128-byte aligned), completing on `bar` (tile::gather4). Rows outside
// the tensor are filled with zeros.
__device__ __forceinline__ void gather4_g2s(void *dst, const CUtensorMap *map, int x, int r0,
                                            int r1, int r2, int r3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1),
          "r"(r2), "r"(r3), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace spmm
