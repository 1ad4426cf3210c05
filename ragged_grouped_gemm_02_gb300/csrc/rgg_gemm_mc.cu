// 128-row 1-CTA tiles on clusters of two CTAs sharing one operand of each
// tile pair through TMA multicast (rgg_gemm_mc.cuh).
#include "rgg_gemm_mc.cuh"
#include "rgg_internal.h"

namespace rgg {

template <int BN, int kEpi = kEpiPlain, bool kFp8 = false>
static cudaError_t launch_mc_instance(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                      const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    auto kernel = grouped_gemm_mc_kernel<BN, kEpi, kFp8>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kernel<<<grid, cta_threads<kEpi, kFp8>(), smem, stream>>>(tmap_x, tmap_x64, tmap_w, args);
    return cudaGetLastError();
}

cudaError_t launch_gemm_mc(int kind, int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                           const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (grid % 2 != 0) return cudaErrorInvalidValue;
    switch (kind) {
        case kMcPlain:
            if (bn == 128) return launch_mc_instance<128>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
            if (bn == 256) return launch_mc_instance<256>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
            return cudaErrorInvalidValue;
        case kMcSwiGLU:
            if (bn == 256)
                return launch_mc_instance<256, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
            return cudaErrorInvalidValue;
        case kMcFp8:
            if (bn == 256)
                return launch_mc_instance<256, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rgg
