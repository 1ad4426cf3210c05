// Grouped GEMM with the token gather fused into the A loads: routed row i of
// the grouped operand is read from token row_index[i] of an ungrouped token
// matrix by TMA tile::gather4 copies, for the plain and the fused gate-up
// epilogues, 64- or 128-row tiles.
#include "rgg_gemm_launch.cuh"

namespace rgg {

cudaError_t launch_gemm_gather(bool swiglu, int bm, int bn, int grid, size_t smem, cudaStream_t stream,
                               const CUtensorMap& tmap_tok, const CUtensorMap& tmap_w, const GemmArgs& args) {
    const CUtensorMap& t = tmap_tok;
    constexpr int G = kGatherTma;
    if (swiglu) {
        if (bm == 128 && bn == 256)
            return launch_gemm_instance<128, 256, kEpiSwiGLU, false, G>(grid, smem, stream, t, t, tmap_w, args);
        if (bm == 128 && bn == 128)
            return launch_gemm_instance<128, 128, kEpiSwiGLU, false, G>(grid, smem, stream, t, t, tmap_w, args);
        if (bm == 64 && bn == 256)
            return launch_gemm_instance<64, 256, kEpiSwiGLU, false, G>(grid, smem, stream, t, t, tmap_w, args);
        if (bm == 64 && bn == 128)
            return launch_gemm_instance<64, 128, kEpiSwiGLU, false, G>(grid, smem, stream, t, t, tmap_w, args);
        return cudaErrorInvalidValue;
    }
    if (bm == 128 && bn == 256)
        return launch_gemm_instance<128, 256, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    if (bm == 128 && bn == 192)
        return launch_gemm_instance<128, 192, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    if (bm == 128 && bn == 128)
        return launch_gemm_instance<128, 128, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    if (bm == 64 && bn == 256)
        return launch_gemm_instance<64, 256, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    if (bm == 64 && bn == 192)
        return launch_gemm_instance<64, 192, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    if (bm == 64 && bn == 128)
        return launch_gemm_instance<64, 128, kEpiPlain, false, G>(grid, smem, stream, t, t, tmap_w, args);
    return cudaErrorInvalidValue;
}

}  // namespace rgg
