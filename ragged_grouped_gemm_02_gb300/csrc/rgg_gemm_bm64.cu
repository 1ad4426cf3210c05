// 64-row tiles (tcgen05 M = 64, cta_group::1) for experts that average 64
// rows or fewer ("Pearl's grouped GEMM kernel for MoE models, explained",
// "Four changes, three of them measured"): half the activation stage, so the
// shared-memory ring holds more weight bytes in flight.
#include "rgg_gemm_launch.cuh"

namespace rgg {

cudaError_t launch_gemm_bm64(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    switch (bn) {
        case 128: return launch_gemm_instance<64, 128>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 192: return launch_gemm_instance<64, 192>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        case 256: return launch_gemm_instance<64, 256>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rgg
