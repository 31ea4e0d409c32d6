// STREAM family, host side: lane shape, range count, the open-row workspace
// and dispatch by reduction. The kernels are in stream.cuh; the per-entry
// row ids are the plan's (gather_prepare).
#include "stream.cuh"

namespace spmm {

int stream_lanes(int64_t N) {
    if (N % 4 != 0 || N <= 32) return 0;
    return N / 4 > 16 ? 32 : 16;
}

int64_t stream_ranges(int64_t nnz, int num_sms, int lanes, int64_t tiles_y) {
    // two waves of the resident warps, shared among the column tiles, each
    // warp walking 32 / lanes ranges; at least 16 entries a range
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t warps = std::max<int64_t>(
        1, 2 * sms * (kStThreads / kWarp) * kStMinBlocks / std::max<int64_t>(1, tiles_y));
    const int64_t r = warps * (kWarp / std::max(1, lanes));
    return std::max<int64_t>(1, std::min<int64_t>(r, nnz / 16));
}

size_t stream_workspace(int64_t ranges, int64_t tiles_y, int lanes, int reduce) {
    const size_t meta = ((size_t)ranges * sizeof(int4) + 255) / 256 * 256;
    const size_t vals = (size_t)tiles_y * (size_t)ranges * 2 * 4 * (size_t)lanes * 4;
    return meta + (reduce == SPMM_MAX ? 2 * vals : vals);
}

cudaError_t launch_stream(const RunArgs &a_in, int reduce, bool has_val, int lanes,
                          int64_t ranges, int tiles_y, cudaStream_t s) {
    RunArgs a = a_in;
    if (!a.ga_rid || ranges < 1 || (lanes != 16 && lanes != 32)) return cudaErrorInvalidValue;
    // the mean runs as the sum kernel with a final 1/d (mean_scale)
    if (reduce == SPMM_MEAN) {
        a.mean = 1;
        reduce = SPMM_SUM;
    }
    a.seg_warps = (int32_t)ranges;
    if (reduce == SPMM_MAX) return launch_stream_red<SPMM_MAX>(a, lanes, has_val, tiles_y, s);
    return launch_stream_red<SPMM_SUM>(a, lanes, has_val, tiles_y, s);
}

}  // namespace spmm
