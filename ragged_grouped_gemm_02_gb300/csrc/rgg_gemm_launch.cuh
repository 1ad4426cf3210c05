// rgg_gemm_launch.cuh -- the host-side launch of one grouped_gemm_kernel
// instantiation (included by the per-BM translation units).
#pragma once

#include "rgg_internal.h"

namespace rgg {

template <int BM, int BN, int kEpi = kEpiPlain, bool kFp8 = false, int kGather = kGatherNone>
cudaError_t launch_gemm_instance(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                 const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    auto kernel = grouped_gemm_kernel<BM, BN, kEpi, kFp8, kGather>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_chained(kernel, grid, cta_threads<kEpi, kFp8>(), smem, stream, tmap_x, tmap_x64, tmap_w, args);
}

}  // namespace rgg
