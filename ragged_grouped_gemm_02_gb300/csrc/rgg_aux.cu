// rgg_aux.cu -- small kernels around the GEMM: the tile-list export (the
// worklog's descriptor list, "Grouped GEMM for Imbalanced Experts on
// Blackwell: A WIP Worklog" section 2, in list order or in the order a walk
// visits it, built by the same device code the GEMM kernels walk), a bare
// offsets check and the two-pass gather's row copy.
#include "rgg_internal.h"

namespace rgg {

// Entry p of the output is the tile at walk position p under `walk_order`
// (0: the flat list itself), decoded by walk_decode exactly as the GEMM
// kernels do: persistent CTA (or CTA pair) c visits positions c, c + grid, ...
__global__ void __launch_bounds__(256) export_tiles_kernel(const int32_t* __restrict__ offsets, int E,
                                                           int64_t M_tot, int N, int BM, int BN, int walk_order,
                                                           int32_t* __restrict__ desc, int64_t cap,
                                                           int32_t* __restrict__ n_tiles,
                                                           int32_t* __restrict__ status) {
    extern __shared__ int32_t sm_export[];
    int32_t* s_off = sm_export;
    int32_t* s_pre = sm_export + (E + 1);
    int32_t* s_order = sm_export + 2 * (E + 1);  // walk order 3 only
    int32_t* s_spre = sm_export + 3 * (E + 1);
    if (!load_and_check_offsets(offsets, s_off, E, M_tot)) {
        if (threadIdx.x == 0) {
            *n_tiles = -1;
            atomicCAS(status, 0, kStatusBadOffsets);
        }
        return;
    }
    const int nN = (N + BN - 1) / BN;
    if ((threadIdx.x >> 5) == 0) build_tile_prefix_warp(s_off, s_pre, E, BM, nN);
    __syncthreads();
    const int32_t T = s_pre[E];
    if (walk_order == 3) build_size_order(s_off, s_order, s_spre, E, BM, nN);
    const int32_t WS = walk_stride_for(T);
    if (threadIdx.x == 0) {
        *n_tiles = T;
        if (static_cast<int64_t>(T) > cap) atomicCAS(status, 0, kStatusCapacity);
    }
    const int64_t limit = static_cast<int64_t>(T) < cap ? static_cast<int64_t>(T) : cap;
    for (int64_t t = threadIdx.x; t < limit; t += blockDim.x) {
        const TileCoord c =
            walk_decode(s_off, s_pre, s_order, s_spre, E, BM, BN, nN, T, walk_order, WS, static_cast<int32_t>(t));
        desc[4 * t + 0] = c.expert;
        desc[4 * t + 1] = c.row0;
        desc[4 * t + 2] = c.rows;
        desc[4 * t + 3] = c.col0;
    }
}

__global__ void __launch_bounds__(256) validate_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                                               int64_t M_tot, int32_t* __restrict__ status) {
    extern __shared__ int32_t sm_validate[];
    if (!load_and_check_offsets(offsets, sm_validate, E, M_tot) && threadIdx.x == 0)
        atomicCAS(status, 0, kStatusBadOffsets);
}

cudaError_t launch_export_tiles(const int32_t* offsets, int E, int64_t M_tot, int N, int bm, int bn,
                                int walk_order, int32_t* desc, int64_t cap, int32_t* n_tiles, int32_t* status,
                                cudaStream_t stream) {
    const size_t smem = (walk_order == 3 ? 4u : 2u) * 4u * static_cast<size_t>(E + 1);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(export_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    export_tiles_kernel<<<1, 256, smem, stream>>>(offsets, E, M_tot, N, bm, bn, walk_order, desc, cap, n_tiles,
                                                  status);
    return cudaGetLastError();
}

// Two-pass token gather, first pass: Xg[i, :] = X_tok[row_index[i], :] for
// the routed rows i in [off[0], off[E]), so that the grouped product can then
// read Xg with whole-tile TMA boxes.  One warp copies one row at a time in
// 16-byte pieces, four loads in flight per lane before their stores.  An
// index outside [0, T) is reported (RGG_ERR_BAD_ROW_INDEX) and token 0 is
// copied in its place, as in the fused gather.  Offsets are only clamped to
// [0, M_tot] here; the GEMM that follows validates them.
__global__ void __launch_bounds__(kGatherRowsThreads) gather_rows_kernel(
    const uint4* __restrict__ xtok, const int32_t* __restrict__ row_index, const int32_t* __restrict__ offsets,
    int E, int64_t M_tot, int64_t T, int kchunks, uint4* __restrict__ xg, int32_t* status) {
    int64_t begin = offsets[0], end = offsets[E];
    begin = begin < 0 ? 0 : (begin > M_tot ? M_tot : begin);
    end = end < begin ? begin : (end > M_tot ? M_tot : end);
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t i = begin + warp; i < end; i += nwarps) {
        int32_t tok = __ldg(row_index + i);
        if (tok < 0 || tok >= T) {
            if (lane == 0) atomicCAS(status, 0, kStatusBadRowIndex);
            tok = 0;
        }
        const uint4* src = xtok + static_cast<int64_t>(tok) * kchunks;
        uint4* dst = xg + i * kchunks;
        int c = lane;
        for (; c + 96 < kchunks; c += 128) {
            const uint4 v0 = __ldg(src + c), v1 = __ldg(src + c + 32), v2 = __ldg(src + c + 64),
                        v3 = __ldg(src + c + 96);
            dst[c] = v0;
            dst[c + 32] = v1;
            dst[c + 64] = v2;
            dst[c + 96] = v3;
        }
        for (; c < kchunks; c += 32) dst[c] = __ldg(src + c);
    }
}

cudaError_t launch_gather_rows(const void* xtok, const int32_t* row_index, const int32_t* offsets, int E,
                               int64_t M_tot, int64_t T, int K, void* xg, int num_sms, int32_t* status,
                               cudaStream_t stream) {
    const int64_t want = (M_tot + kGatherRowsThreads / 32 - 1) / (kGatherRowsThreads / 32);
    const int grid = static_cast<int>(want < 1 ? 1 : (want > 4LL * num_sms ? 4LL * num_sms : want));
    gather_rows_kernel<<<grid, kGatherRowsThreads, 0, stream>>>(static_cast<const uint4*>(xtok), row_index, offsets,
                                                                 E, M_tot, T, K / 8, static_cast<uint4*>(xg), status);
    return cudaGetLastError();
}

cudaError_t launch_validate_offsets(const int32_t* offsets, int E, int64_t M_tot, int32_t* status,
                                    cudaStream_t stream) {
    const size_t smem = 4u * static_cast<size_t>(E + 1);
    validate_offsets_kernel<<<1, 256, smem, stream>>>(offsets, E, M_tot, status);
    return cudaGetLastError();
}

}  // namespace rgg
