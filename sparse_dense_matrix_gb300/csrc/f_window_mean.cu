// WINDOW kernel instantiations for the mean reduction.
#include "window.cuh"

namespace spmm {
template cudaError_t launch_window_red<SPMM_MEAN>(const RunArgs &, const WinShape &,
                                              const CUtensorMap &, bool, bool, int, int,
                                              cudaStream_t);
}  // namespace spmm
