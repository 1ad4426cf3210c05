// 256-row tiles on a CTA pair (tcgen05 cta_group::2, clusters of two CTAs).
#include "rgg_gemm_2cta.cuh"
#include "rgg_internal.h"

namespace rgg {

template <int BN, int kEpi = kEpiPlain, bool kFp8 = false>
static cudaError_t launch_pair_instance(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                        const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w,
                                        const GemmArgs& args) {
    auto kernel = grouped_gemm_pair_kernel<BN, kEpi, kFp8>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kernel<<<grid, 64 + 32 * pair_epilogue_warps<kEpi, kFp8>(), smem, stream>>>(tmap_x, tmap_x64, tmap_w, args);
    return cudaGetLastError();
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

// FP8 (E4M3) operands with per-row / per-column scales on CTA pairs: `bn` is 256.
cudaError_t launch_gemm_pair_fp8(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                 const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (grid % 2 != 0 || bn != 256) return cudaErrorInvalidValue;
    return launch_pair_instance<256, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
}

}  // namespace rgg
