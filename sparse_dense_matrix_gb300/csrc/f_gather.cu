// GATHER family, host side: the plan's per-entry row array, the grid, the
// open-row workspace, B's tensor map and dispatch by reduction. The kernels
// are in gather.cuh.
#include <cstring>

#include <cudaTypedefs.h>

#include "gather.cuh"

namespace spmm {

// row id of every stored entry: a warp per row, lanes over the row's entries
__global__ void __launch_bounds__(256) k_ga_rid(const int32_t *__restrict__ rowptr, int64_t M,
                                                int32_t *__restrict__ rid) {
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; i < M;
         i += warps) {
        const int b = rowptr[i], e = rowptr[i + 1];
        for (int p = b + lane; p < e; p += kWarp) rid[p] = (int32_t)i;
    }
}

int gather_tile(int64_t N) { return N % 256 == 0 ? 256 : N % 128 == 0 ? 128 : 0; }

int64_t gather_ctas(int64_t nnz, int num_sms, int64_t tiles_y) {
    // two CTAs per SM (96 KB rings), shared among the column tiles; never
    // more CTAs than entries, so that every range holds at least one
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t ctas = std::max<int64_t>(1, 2 * sms / std::max<int64_t>(1, tiles_y));
    return std::max<int64_t>(1, std::min<int64_t>(ctas, nnz));
}

size_t gather_workspace(int64_t ctas, int64_t tiles_y, int ct, int reduce) {
    const size_t meta = ((size_t)ctas * sizeof(int4) + 255) / 256 * 256;
    const size_t vals = (size_t)tiles_y * (size_t)ctas * 2 * (size_t)ct * 4;
    return meta + (reduce == SPMM_MAX ? 2 * vals : vals);
}

cudaError_t gather_prepare(Plan *p, cudaStream_t s) {
    if (p->ga_rid) return cudaSuccess;
    int32_t *rid = nullptr;
    cudaError_t e = cudaMalloc((void **)&rid, sizeof(int32_t) * (size_t)std::max<int64_t>(1, p->nnz));
    if (e != cudaSuccess) return e;
    const int64_t blocks = std::min<int64_t>((p->M + 7) / 8, (int64_t)std::max(1, p->num_sms) * 8);
    k_ga_rid<<<(unsigned)std::max<int64_t>(1, blocks), 256, 0, s>>>(p->rowptr, p->M, rid);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaFree(rid);
        return e;
    }
    p->ga_rid = rid;
    p->ga_bytes = (int64_t)sizeof(int32_t) * p->nnz;
    return cudaSuccess;
}

void gather_free(Plan *p) {
    if (p->ga_rid) cudaFree(p->ga_rid);
    p->ga_rid = nullptr;
    p->ga_bytes = 0;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// B as a 2-D tensor (N columns, K rows) in boxes of one row of ct columns:
// the shape tile::gather4 copies (four such rows per instruction)
cudaError_t encode_rows(const RunArgs &a, int ct, CUtensorMap *map) {
    std::memset(map, 0, sizeof(*map));
    if (!g_encode) {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
    const cuuint32_t box[2] = {(cuuint32_t)ct, 1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.B), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_gather(const RunArgs &a_in, int reduce, bool has_val, int ctas, int tiles_y,
                          cudaStream_t s) {
    RunArgs a = a_in;
    const int ct = gather_tile(a.N);
    if (!ct || (int64_t)ct * tiles_y != a.N || ctas < 1 || !a.ga_rid) return cudaErrorInvalidValue;
    // the mean runs as the sum kernel with a final 1/d (mean_scale)
    if (reduce == SPMM_MEAN) {
        a.mean = 1;
        reduce = SPMM_SUM;
    }
    a.seg_warps = ctas;
    CUtensorMap map;
    cudaError_t e = encode_rows(a, ct, &map);
    if (e != cudaSuccess) return e;
    if (reduce == SPMM_MAX) return launch_gather_red<SPMM_MAX>(a, map, ct, has_val, ctas, tiles_y, s);
    return launch_gather_red<SPMM_SUM>(a, map, ct, has_val, ctas, tiles_y, s);
}

}  // namespace spmm
