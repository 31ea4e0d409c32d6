// Diagnostic: the bounded-wait path that every spin-wait of the library
// relies on, exercised on purpose. One warp waits on an mbarrier that nothing
// arrives on; the wait gives up after the given time, records the timeout in
// the plan's error words and returns, so the kernel ends and the context
// stays usable. No fault, no trap, no unbounded loop.
#include "common.cuh"
#include "tma.cuh"

namespace spmm {
namespace {

__global__ void k_wait_nobody(int32_t *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);            // one arrival expected; none is ever made
        mbar_init_fence();
    }
    __syncthreads();
    mbar_wait(&bar, 0u, err, limit_ns);
}

}  // namespace
}  // namespace spmm

extern "C" spmm_status spmm_check_wait_timeout(spmm_plan_t plan, int64_t limit_us, void *stream) {
    using namespace spmm;
    if (!plan || limit_us < 1 || limit_us > 10 * 1000 * 1000) return SPMM_ERR_INVALID_ARG;
    Plan *p = reinterpret_cast<Plan *>(plan);
    cudaStream_t s = (cudaStream_t)stream;
    k_wait_nobody<<<1, kWarp, 0, s>>>(p->err, (uint64_t)limit_us * 1000u);
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SPMM_ERR_OOM : SPMM_ERR_CUDA;
    return spmm_plan_sync(plan, stream);
}
