// SEGMENT family, sum instantiation (see segment.cuh).
#include "segment.cuh"

namespace spmm {
template cudaError_t launch_segment_red<SPMM_SUM>(const RunArgs &, int, int, bool, int, int,
                                                  cudaStream_t);
}  // namespace spmm
