// 128-row tiles (tcgen05 M = 128, cta_group::1): one TMEM lane per tile row.
#include "rgg_gemm_launch.cuh"

namespace rgg {

cudaError_t launch_gemm_bm128(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    switch (bn) {
        case 128: return launch_gemm_instance<128, 128>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 192: return launch_gemm_instance<128, 192>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 256: return launch_gemm_instance<128, 256>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rgg
