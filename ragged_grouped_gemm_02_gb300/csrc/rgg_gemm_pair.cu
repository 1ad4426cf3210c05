// 256-row tiles on a CTA pair (tcgen05 cta_group::2, clusters of two CTAs).
#include "rgg_gemm_2cta.cuh"
#include "rgg_internal.h"

namespace rgg {

template <int BN, int kEpi = kEpiPlain>
static cudaError_t launch_pair_instance(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                        const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w,
                                        const GemmArgs& args) {
    auto kernel = grouped_gemm_pair_kernel<BN, kEpi>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_chained(kernel, grid, 64 + 32 * pair_epilogue_warps<kEpi>(), smem, stream, tmap_x, tmap_x64, tmap_w,
                          args);
}

cudaError_t launch_gemm_pair(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (grid % 2 != 0) return cudaErrorInvalidValue;
    switch (bn) {
        case 128: return launch_pair_instance<128>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 256: return launch_pair_instance<256>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        default: return cudaErrorInvalidValue;
    }
}

// The fused gate-up + SiLU epilogue on CTA pairs: `bn` (the MMA width, twice
// the output columns per tile) is 128 or 256.
cudaError_t launch_gemm_pair_swiglu(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                    const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (grid % 2 != 0) return cudaErrorInvalidValue;
    switch (bn) {
        case 128: return launch_pair_instance<128, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 256: return launch_pair_instance<256, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rgg
