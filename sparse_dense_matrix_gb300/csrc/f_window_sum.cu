// WINDOW kernel instantiations for the sum reduction.
#include "window.cuh"

namespace spmm {
template cudaError_t launch_window_red<SPMM_SUM>(const RunArgs &, const WinShape &,
                                              const CUtensorMap &, bool, bool, int, int,
                                              cudaStream_t);
}  // namespace spmm
