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
// block must call this; returns the same answer in every thread.
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

// The same prefix over one class of experts: expert e counts only when
// lo <= m_e < hi (its tiles of BM rows), the others add no tiles.  Used by the
// mixed launch, whose CTA pairs take the experts of at least `pair_min_rows`
// rows in 256-row tiles and whose 1-CTA kernel takes the rest in 128-row
// tiles, each class with its own flat list in the worklog's order.
__device__ __forceinline__ void build_class_prefix_warp(const int32_t* s_off, int32_t* s_pre, int E, int BM,
                                                        int n_tiles_n, int32_t lo, int32_t hi) {
    const int lane = threadIdx.x & 31;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per);
    const int e1 = min(E, e0 + per);
    auto tiles = [&](int e) -> int32_t {
        const int32_t m = s_off[e + 1] - s_off[e];
        return (m >= lo && m < hi) ? ((m + BM - 1) / BM) * n_tiles_n : 0;
    };
    int32_t local = 0;
    for (int e = e0; e < e1; ++e) local += tiles(e);
    int32_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    int32_t run = incl - local;
    for (int e = e0; e < e1; ++e) {
        s_pre[e] = run;
        run += tiles(e);
    }
    if (lane == 31) s_pre[E] = incl;
}

// Decode flat tile t (0 <= t < s_pre[E]).  The expert is the last e with
// s_pre[e] <= t, which skips empty experts because they add no tiles.
// `n_major` (walk order 4) visits an expert's tiles N tile by N tile (all M
// tiles of one weight panel, then the next panel) instead of M tile by M tile;
// the set of tiles is the same.
__device__ __forceinline__ TileCoord decode_tile(const int32_t* s_off, const int32_t* s_pre, int E, int BM,
                                                 int BN, int n_tiles_n, int32_t t, bool n_major = false) {
    int lo = 0, hi = E;  // s_pre[lo] <= t < s_pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int32_t local = t - s_pre[lo];
    const int32_t m_e = s_off[lo + 1] - s_off[lo];
    int32_t mt, nt;
    if (n_major) {
        const int32_t nm = (m_e + BM - 1) / BM;
        nt = local / nm;
        mt = local - nt * nm;
    } else {
        mt = local / n_tiles_n;
        nt = local - mt * n_tiles_n;
    }
    TileCoord c;
    c.expert = lo;
    c.row0 = s_off[lo] + mt * BM;
    c.rows = min(BM, m_e - mt * BM);
    c.col0 = nt * BN;
    return c;
}

// The order in which a persistent CTA visits the flat list.  Every order is a
// permutation of [0, T), so the result does not depend on it; it only changes
// which tiles run side by side on the GPU.  0: list order (CTA c takes
// c, c + grid, ...).  1: front/back interleave (even walk positions from the
// front of the list, odd ones from the back), which pairs the big experts at
// one end of an expert-sorted list with the small ones at the other.
// 2: strided scatter p -> p * s mod T with a prime s that does not divide T.
// (3 is the size-sorted walk below; 4 is list order with each expert's tiles
// taken N-major, see decode_tile.)
__device__ __forceinline__ int32_t walk_stride_for(int32_t T) {
    const int32_t primes[4] = {7919, 6841, 5009, 1009};
    for (int i = 0; i < 4; ++i)
        if (T % primes[i] != 0) return primes[i];
    return 1;
}

__device__ __forceinline__ int32_t walk_tile(int32_t p, int32_t T, int order, int32_t stride) {
    if (order == 1 || order == 3) return (p & 1) ? T - 1 - (p >> 1) : (p >> 1);
    if (order == 2) return static_cast<int32_t>((static_cast<int64_t>(p) * stride) % T);
    return p;
}

// Walk order 3 walks the tiles of the experts sorted by row count (largest
// first, ties by index) with the front/back interleave, so that tiles of big
// experts (weights reused from L2, MMA-heavy) run beside tiles of small ones
// (weights streamed from HBM).  Every thread of the block calls this; it
// fills s_order (rank -> expert) and the tile prefix over ranks s_spre[0..E].
constexpr int kMaxSortedExperts = 256;

__device__ __forceinline__ void build_size_order(const int32_t* s_off, int32_t* s_order, int32_t* s_spre, int E,
                                                 int BM, int n_tiles_n) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t m = s_off[e + 1] - s_off[e];
        int rank = 0;
        for (int f = 0; f < E; ++f) {
            const int32_t mf = s_off[f + 1] - s_off[f];
            rank += (mf > m || (mf == m && f < e)) ? 1 : 0;
        }
        s_order[rank] = e;
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        const int lane = threadIdx.x & 31;
        const int per = (E + 31) / 32;
        const int r0 = min(E, lane * per);
        const int r1 = min(E, r0 + per);
        int32_t local = 0;
        for (int r = r0; r < r1; ++r) {
            const int e = s_order[r];
            local += ((s_off[e + 1] - s_off[e] + BM - 1) / BM) * n_tiles_n;
        }
        int32_t incl = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        int32_t run = incl - local;
        for (int r = r0; r < r1; ++r) {
            s_spre[r] = run;
            const int e = s_order[r];
            run += ((s_off[e + 1] - s_off[e] + BM - 1) / BM) * n_tiles_n;
        }
        if (lane == 31) s_spre[E] = incl;
    }
    __syncthreads();
}

// Decode position t of the size-sorted sequence (0 <= t < s_spre[E]).
__device__ __forceinline__ TileCoord decode_sorted_tile(const int32_t* s_off, const int32_t* s_order,
                                                        const int32_t* s_spre, int E, int BM, int BN, int n_tiles_n,
                                                        int32_t t) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_spre[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int e = s_order[lo];
    const int32_t local = t - s_spre[lo];
    const int32_t mt = local / n_tiles_n;
    const int32_t nt = local - mt * n_tiles_n;
    const int32_t m_e = s_off[e + 1] - s_off[e];
    TileCoord c;
    c.expert = e;
    c.row0 = s_off[e] + mt * BM;
    c.rows = min(BM, m_e - mt * BM);
    c.col0 = nt * BN;
    return c;
}

// The tile visited at walk position p (0 <= p < T) under walk order WO (WS =
// walk_stride_for(T)): the decode every GEMM kernel and the walk export use.
// s_order / s_spre are read only for the size-sorted walk (3).
__device__ __forceinline__ TileCoord walk_decode(const int32_t* s_off, const int32_t* s_pre, const int32_t* s_order,
                                                 const int32_t* s_spre, int E, int BM, int BN, int n_tiles_n,
                                                 int32_t T, int WO, int32_t WS, int32_t p) {
    const int32_t t = walk_tile(p, T, WO, WS);
    if (WO == 3) return decode_sorted_tile(s_off, s_order, s_spre, E, BM, BN, n_tiles_n, t);
    return decode_tile(s_off, s_pre, E, BM, BN, n_tiles_n, t, WO == 4);
}

}  // namespace rgg
