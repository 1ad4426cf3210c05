// FP8 (E4M3) operands, tcgen05.mma kind::f8f6f4, fp32 accumulator, per-row
// and per-(expert, column) scales applied in the epilogue.
#include "rgg_gemm_launch.cuh"

namespace rgg {

cudaError_t launch_gemm_fp8(int bm, int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                            const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args) {
    if (bm == 128 && bn == 256)
        return launch_gemm_instance<128, 256, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 128 && bn == 128)
        return launch_gemm_instance<128, 128, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 64 && bn == 256)
        return launch_gemm_instance<64, 256, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    if (bm == 64 && bn == 128)
        return launch_gemm_instance<64, 128, kEpiPlain, true>(grid, smem, stream, tmap_x, tmap_x64, tmap_w, args);
    return cudaErrorInvalidValue;
}

}  // namespace rgg
