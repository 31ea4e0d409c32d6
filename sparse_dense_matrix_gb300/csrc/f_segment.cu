// SEGMENT family, host side: grid size, the workspace of the open-row
// partials, and dispatch by reduction. The kernels are in segment.cuh.
#include "segment.cuh"

namespace spmm {

int64_t segment_warps(int64_t n_tiles, int num_sms, int64_t tiles_y) {
    // one CTA of kSegWarps warps per SM (its shared memory takes most of an
    // SM), shared among the column tiles; never more warps than tiles
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t ctas = std::max<int64_t>(1, sms / std::max<int64_t>(1, tiles_y));
    return std::max<int64_t>(1, std::min<int64_t>(ctas * kSegWarps, n_tiles));
}

size_t segment_workspace(int64_t seg_warps, int64_t tiles_y, int lanes, int chunks, int reduce) {
    const size_t cw = 4 * (size_t)lanes * (size_t)chunks;
    const size_t meta = ((size_t)seg_warps * sizeof(int4) + 255) / 256 * 256;
    const size_t vals = (size_t)tiles_y * (size_t)seg_warps * 2 * cw * 4;
    return meta + (reduce == SPMM_MAX ? 2 * vals : vals);
}

cudaError_t launch_segment(const RunArgs &a_in, int lanes, int chunks, int reduce, bool has_val,
                           int tiles_y, cudaStream_t s) {
    RunArgs a = a_in;
    // the mean runs as the sum kernel with a final 1/d (mean_scale)
    if (reduce == SPMM_MEAN) {
        a.mean = 1;
        reduce = SPMM_SUM;
    }
    const int ctas_x = (int)((a.seg_warps + kSegWarps - 1) / kSegWarps);
    if (reduce == SPMM_MAX)
        return launch_segment_red<SPMM_MAX>(a, lanes, chunks, has_val, ctas_x, tiles_y, s);
    return launch_segment_red<SPMM_SUM>(a, lanes, chunks, has_val, ctas_x, tiles_y, s);
}

}  // namespace spmm
