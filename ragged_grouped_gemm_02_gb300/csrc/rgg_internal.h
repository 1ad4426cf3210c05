// rgg_internal.h -- launch entry points shared between the C ABI layer
// (rgg_api.cu) and the translation units that instantiate the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "rgg.h"
#include "rgg_gemm.cuh"

namespace rgg {

// Every GEMM kernel is launched with programmatic stream serialisation: it
// may become resident while the kernel ahead of it on the stream is still
// running (its CTAs take SMs as that kernel's CTAs exit), and waits on the
// device (griddepcontrol.wait) before its first global memory access.  Back
// to back launches then hide most of the launch and CTA-dispatch latency.
// Ahead of a copy or a memset, or a kernel launched without the attribute,
// the launch is ordered as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), int grid, int threads, size_t smem, cudaStream_t stream,
                           Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// Grouped GEMM kernels, one translation unit per BM.  `bn` is 128, 192 or
// 256.  tmap_x64 is X with a 64-row box (tail tiles of 128-row kernels).
// Returns cudaErrorInvalidValue for a shape with no instantiation.
cudaError_t launch_gemm_bm128(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                              const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);
cudaError_t launch_gemm_bm64(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);

// Fused gate-up + SiLU (kEpiSwiGLU): `bm` is 64 or 128, `bn` (the MMA width,
// twice the output columns per tile) is 128 or 256; tmap_w spans 2N columns.
cudaError_t launch_gemm_swiglu(int bm, int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                               const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);

// FP8 (E4M3) operands with per-row / per-column scales: `bm` 64 or 128, `bn`
// 128 or 256; the tensor maps are over bytes with 128-byte boxes.
cudaError_t launch_gemm_fp8(int bm, int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                            const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);

// Token gather fused into the A loads (TMA tile::gather4): tmap_tok is the
// token matrix [T, K] with a one-row box.  `swiglu` selects the fused gate-up
// epilogue (then `bn` is the MMA width, 128 or 256); otherwise `bn` is 128,
// 192 or 256.  `bm` is 64 or 128.
cudaError_t launch_gemm_gather(bool swiglu, int bm, int bn, int grid, size_t smem, cudaStream_t stream,
                               const CUtensorMap& tmap_tok, const CUtensorMap& tmap_w, const GemmArgs& args);

// First pass of the two-pass gather: Xg[i] = X_tok[row_index[i]] for the rows
// [off[0], off[E]) (clamped to [0, M_tot]).  xtok and xg are 16-byte aligned
// bf16 [T, K] and [M_tot, K]; K is a multiple of 8.
constexpr int kGatherRowsThreads = 512;
cudaError_t launch_gather_rows(const void* xtok, const int32_t* row_index, const int32_t* offsets, int E,
                               int64_t M_tot, int64_t T, int K, void* xg, int num_sms, int32_t* status,
                               cudaStream_t stream);

// CTA-pair kernel (256-row tiles, clusters of two): `bn` is 128 or 256 and
// `grid` is even.
cudaError_t launch_gemm_pair(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);
// The same with the fused gate-up + SiLU epilogue (tmap_w spans 2N columns; tail tiles stay M = 256).
cudaError_t launch_gemm_pair_swiglu(int bn, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& tmap_x,
                                    const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w, const GemmArgs& args);

// The mixed launch: the pair kernel (pair_grid CTAs, even; may be 0) and,
// after it with programmatic stream serialisation, the 1-CTA kernel
// (single_grid CTAs; may be 0), both 256-column tiles claiming from the two
// counters at pair_args.sched (zeroed by the caller before the launch).
cudaError_t launch_gemm_mixed(int pair_grid, size_t pair_smem, const GemmArgs& pair_args, int single_grid,
                              size_t single_smem, const GemmArgs& single_args, cudaStream_t stream,
                              const CUtensorMap& tmap_x, const CUtensorMap& tmap_x64, const CUtensorMap& tmap_w);
// The same with the fused gate-up + SiLU epilogue (tmap_w spans 2N columns;
// 128 output columns per tile; pair tail tiles stay 256 rows).
cudaError_t launch_gemm_mixed_swiglu(int pair_grid, size_t pair_smem, const GemmArgs& pair_args, int single_grid,
                                     size_t single_smem, const GemmArgs& single_args, cudaStream_t stream,
                                     const CUtensorMap& tmap_x, const CUtensorMap& tmap_x64,
                                     const CUtensorMap& tmap_w);

// The flat tile list written out by the same device code the GEMM uses, in
// list order (walk_order 0) or in the order walk_order visits it.
cudaError_t launch_export_tiles(const int32_t* offsets, int E, int64_t M_tot, int N, int bm, int bn,
                                int walk_order, int32_t* desc, int64_t cap, int32_t* n_tiles, int32_t* status,
                                cudaStream_t stream);

// Host helpers defined in rgg_api.cu: the thread-local text behind
// rgg_last_cuda_error().
rgg_status host_cuda_failure(cudaError_t err, const char* what);
void host_set_last_error(const char* what);

// The argument checks of rgg_grouped_gemm (null pointers, sizes, alignment).
rgg_status host_check_gemm_args(const void* X, const void* W, const int32_t* group_offsets, const void* Y, int E,
                                int64_t M_tot, int K, int N);
// Plan, encode and launch rgg_grouped_gemm on the current device for a GPU of
// `num_sms` SMs and `smem_optin` bytes of shared memory per block, recording
// device-detected errors in the device word `status`.  Arguments already
// checked by host_check_gemm_args.
rgg_status host_grouped_gemm(int num_sms, int smem_optin, int32_t* status, const void* X, const void* W,
                             const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N,
                             cudaStream_t stream, const rgg_options* opt);

// Offsets check alone (used when there are no rows to multiply).
cudaError_t launch_validate_offsets(const int32_t* offsets, int E, int64_t M_tot, int32_t* status,
                                    cudaStream_t stream);

}  // namespace rgg
