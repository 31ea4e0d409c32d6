// STREAM family, max instantiation (see stream.cuh).
#include "stream.cuh"

namespace spmm {
template cudaError_t launch_stream_red<SPMM_MAX>(const RunArgs &, int, bool, int, cudaStream_t);
}  // namespace spmm
