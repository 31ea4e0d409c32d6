// SEGMENT family, max instantiation (see segment.cuh).
#include "segment.cuh"

namespace spmm {
template cudaError_t launch_segment_red<SPMM_MAX>(const RunArgs &, int, int, bool, int, int,
                                                  cudaStream_t);
}  // namespace spmm
