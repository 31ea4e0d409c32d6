// STREAM family, sum instantiation (see stream.cuh).
#include "stream.cuh"

namespace spmm {
template cudaError_t launch_stream_red<SPMM_SUM>(const RunArgs &, int, bool, int, cudaStream_t);
}  // namespace spmm
