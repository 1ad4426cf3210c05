// rgg_aux.cu -- small kernels around the GEMM: the tile-list export (the
// worklog's descriptor list, "Grouped GEMM for Imbalanced Experts on
// Blackwell: A WIP Worklog" section 2, built by the same device code the GEMM
// kernel walks) and a bare offsets check.
#include "rgg_internal.h"

namespace rgg {

__global__ void __launch_bounds__(256) export_tiles_kernel(const int32_t* __restrict__ offsets, int E,
                                                           int64_t M_tot, int N, int BM, int BN,
                                                           int32_t* __restrict__ desc, int64_t cap,
                                                           int32_t* __restrict__ n_tiles,
                                                           int32_t* __restrict__ status) {
    extern __shared__ int32_t sm_export[];
    int32_t* s_off = sm_export;
    int32_t* s_pre = sm_export + (E + 1);
    if (!load_and_check_offsets(offsets, s_off, E, M_tot)) {
        if (threadIdx.x == 0) {
            *n_tiles = -1;
            atomicCAS(status, 0, kStatusBadOffsets);
        }
        return;
    }
    const int nN = (N + BN - 1) / BN;
    if ((threadIdx.x >> 5) == 0) build_tile_prefix_warp(s_off, s_pre, E, BM, nN);
    __syncthreads();
    const int32_t T = s_pre[E];
    if (threadIdx.x == 0) {
        *n_tiles = T;
        if (static_cast<int64_t>(T) > cap) atomicCAS(status, 0, kStatusCapacity);
    }
    const int64_t limit = static_cast<int64_t>(T) < cap ? static_cast<int64_t>(T) : cap;
    for (int64_t t = threadIdx.x; t < limit; t += blockDim.x) {
        const TileCoord c = decode_tile(s_off, s_pre, E, BM, BN, nN, static_cast<int32_t>(t));
        desc[4 * t + 0] = c.expert;
        desc[4 * t + 1] = c.row0;
        desc[4 * t + 2] = c.rows;
        desc[4 * t + 3] = c.col0;
    }
}

__global__ void __launch_bounds__(256) validate_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                                               int64_t M_tot, int32_t* __restrict__ status) {
    extern __shared__ int32_t sm_validate[];
    if (!load_and_check_offsets(offsets, sm_validate, E, M_tot) && threadIdx.x == 0)
        atomicCAS(status, 0, kStatusBadOffsets);
}

cudaError_t launch_export_tiles(const int32_t* offsets, int E, int64_t M_tot, int N, int bm, int bn,
                                int32_t* desc, int64_t cap, int32_t* n_tiles, int32_t* status,
                                cudaStream_t stream) {
    const size_t smem = 2u * 4u * static_cast<size_t>(E + 1);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(export_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    export_tiles_kernel<<<1, 256, smem, stream>>>(offsets, E, M_tot, N, bm, bn, desc, cap, n_tiles, status);
    return cudaGetLastError();
}

cudaError_t launch_validate_offsets(const int32_t* offsets, int E, int64_t M_tot, int32_t* status,
                                    cudaStream_t stream) {
    const size_t smem = 4u * static_cast<size_t>(E + 1);
    validate_offsets_kernel<<<1, 256, smem, stream>>>(offsets, E, M_tot, status);
    return cudaGetLastError();
}

}  // namespace rgg
