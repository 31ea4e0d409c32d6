// GATHER family, max instantiation (see gather.cuh).
#include "gather.cuh"

namespace spmm {
template cudaError_t launch_gather_red<SPMM_MAX>(const RunArgs &, const CUtensorMap &, int, bool,
                                                 int, int, cudaStream_t);
}  // namespace spmm
