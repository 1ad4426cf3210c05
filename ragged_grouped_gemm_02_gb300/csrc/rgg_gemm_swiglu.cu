// The fused gate-up projection with SiLU activation (epilogue kEpiSwiGLU):
// 64- or 128-row tiles, MMA width 128 or 256 (= 64 or 128 output columns).
#include "rgg_gemm_launch.cuh"

namespace rgg {

cudaError_t launch_gemm_swiglu(int bm, int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                               const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (bm == 128 && bn == 256)
        return launch_gemm_instance<128, 256, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 128 && bn == 128)
        return launch_gemm_instance<128, 128, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 64 && bn == 256)
        return launch_gemm_instance<64, 256, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 64 && bn == 128)
        return launch_gemm_instance<64, 128, kEpiSwiGLU>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    return cudaErrorInvalidValue;
}

}  // namespace rgg
