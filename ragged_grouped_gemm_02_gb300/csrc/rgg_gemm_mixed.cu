// The mixed launch (rgg_sched.cuh): 256-row tiles of the large experts on CTA
// pairs beside 128-row tiles of the small ones on single CTAs, two kernels on
// disjoint SMs that claim tiles from the same two device counters.
#include "rgg_gemm_2cta.cuh"
#include "rgg_internal.h"

namespace rgg {

template <int kEpi>
static cudaError_t launch_mixed_instance(int pair_grid, size_t pair_smem, const GemmArgs& pair_args, int single_grid,
                                         size_t single_smem, const GemmArgs& single_args, cudaStream_t stream,
                                         const CUtensorMap& tmap_x, const CUtensorMap& tmap_x64,
                                         const CUtensorMap& tmap_w) {
    if (pair_grid < 0 || pair_grid % 2 != 0 || single_grid < 0 || pair_grid + single_grid == 0)
        return cudaErrorInvalidValue;
    if (pair_grid > 0) {
        auto kernel = grouped_gemm_pair_kernel<kMixedBN, kEpi, true>;
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(pair_smem));
        if (err != cudaSuccess) return err;
        err = launch_chained(kernel, pair_grid, 64 + 32 * pair_epilogue_warps<kEpi>(), pair_smem, stream, tmap_x,
                             tmap_x64, tmap_w, pair_args);
        if (err != cudaSuccess) return err;
    }
    if (single_grid > 0) {
        auto kernel = grouped_gemm_kernel<128, kMixedBN, kEpi, false, kGatherNone, true>;
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(single_smem));
        if (err != cudaSuccess) return err;
        // After the pair kernel: starts once every pair CTA has passed its own
        // wait for the work ahead on the stream, so the two kernels share the
        // GPU; it does not wait for the pair kernel before its loads, only
        // before it ends (so the stream's later work sees both done).  Alone
        // (no pair CTAs) it waits first, like every other kernel.
        GemmArgs a = single_args;
        a.pdl_wait_first = pair_grid > 0 ? 0 : 1;
        return launch_chained(kernel, single_grid, cta_threads<kEpi, false>(), single_smem, stream, tmap_x, tmap_x64,
                              tmap_w, a);
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_mixed(int pair_grid, size_t pair_smem, const GemmArgs& pair_args, int single_grid,
                              size_t single_smem, const GemmArgs& single_args, cudaStream_t stream,
                              const CUtensorMap& tmap_x, const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w) {
    return launch_mixed_instance<kEpiPlain>(pair_grid, pair_smem, pair_args, single_grid, single_smem, single_args,
                                            stream, tmap_x, tmap_x64, tmap_w);
}

cudaError_t launch_gemm_mixed_swiglu(int pair_grid, size_t pair_smem, const GemmArgs& pair_args, int single_grid,
                                     size_t single_smem, const GemmArgs& single_args, cudaStream_t stream,
                                     const CUtensorMap& tmap_x, const CUtensorMap& tmap_x64,
                                     const CUtensorMap& tmap_w) {
    return launch_mixed_instance<kEpiSwiGLU>(pair_grid, pair_smem, pair_args, single_grid, single_smem, single_args,
                                             stream, tmap_x, tmap_x64, tmap_w);
}

}  // namespace rgg
