// rgg_tiles.cuh -- the flat tile list, built on the device from the group
// offsets and decoded per tile.
//
// "Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog", section 2
// ("The Grouped Problem and the flat tile list"): all output tiles of all
// experts form one expert-major list; expert e contributes ceil(m_e/BM) M
// tiles times ceil(N/BN) N tiles; tile (e, mt, nt) covers rows
// off[e] + mt*BM .. + min(BM, m_e - mt*BM) and columns nt*BN ..; tiles stop at
// expert boundaries and each tile owns its whole K reduction.  The worklog
// builds this list on the host; here every CTA builds the per-expert tile
// prefix in shared memory from the device-side offsets (the "Grouped GEMM"
// glossary's "fuses group metadata generation into the kernel"), so the
// routed counts never travel to the host and a launch can sit in a CUDA graph.
#pragma once

#include <cstdint>

namespace rgg {

constexpr int kMaxExperts = 4096;

struct TileCoord {
    int32_t expert;
    int32_t row0;
    int32_t rows;
    int32_t col0;
};

// Load off[0..E] into shared memory and check validity:
// 0 <= off[0] <= off[1] <= ... <= off[E] <= M_tot.  Every thread of the
// block must call this; returns the same verdict in every thread.
__device__ __forceinline__ bool load_and_check_offsets(const int32_t* __restrict__ g_off, int32_t* s_off, int E,
                                                       int64_t M_tot) {
    int bad = 0;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int32_t v = g_off[e];
        s_off[e] = v;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        bad |= (s_off[e + 1] < s_off[e]) ? 1 : 0;
    if (threadIdx.x == 0)
        bad |= (s_off[0] < 0 || static_cast<int64_t>(s_off[E]) > M_tot) ? 1 : 0;
    return __syncthreads_or(bad) == 0;
}

// Exclusive prefix of tiles per expert, s_pre[0..E], computed by one warp
// (lane = threadIdx.x & 31 of the calling warp).  Each lane sums a contiguous
// chunk of experts, the warp scans the chunk sums, then each lane writes its
// chunk.  s_pre[E] is the total tile count T.  The caller synchronises the
// block afterwards.
__device__ __forceinline__ void build_tile_prefix_warp(const int32_t* s_off, int32_t* s_pre, int E, int BM,
                                                       int n_tiles_n) {
    const int lane = threadIdx.x & 31;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per);
    const int e1 = min(E, e0 + per);
    int32_t local = 0;
    for (int e = e0; e < e1; ++e) {
        const int32_t m = s_off[e + 1] - s_off[e];
        local += ((m + BM - 1) / BM) * n_tiles_n;
    }
    int32_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    int32_t run = incl - local;
    for (int e = e0; e < e1; ++e) {
        s_pre[e] = run;
        const int32_t m = s_off[e + 1] - s_off[e];
        run += ((m + BM - 1) / BM) * n_tiles_n;
    }
    if (lane == 31) s_pre[E] = incl;
}

// Decode flat tile t (0 <= t < s_pre[E]).  The expert is the last e with
// s_pre[e] <= t, which skips empty experts because they add no tiles.
__device__ __forceinline__ TileCoord decode_tile(const int32_t* s_off, const int32_t* s_pre, int E, int BM,
                                                 int BN, int n_tiles_n, int32_t t) {
    int lo = 0, hi = E;  // s_pre[lo] <= t < s_pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int32_t local = t - s_pre[lo];
    const int32_t mt = local / n_tiles_n;
    const int32_t nt = local - mt * n_tiles_n;
    const int32_t m_e = s_off[lo + 1] - s_off[lo];
    TileCoord c;
    c.expert = lo;
    c.row0 = s_off[lo] + mt * BM;
    c.rows = min(BM, m_e - mt * BM);
    c.col0 = nt * BN;
    return c;
}

}  // namespace rgg
