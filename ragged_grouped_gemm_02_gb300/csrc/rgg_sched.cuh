// rgg_sched.cuh -- the tile claims of the mixed launch: CTA pairs for large
// experts beside 1-CTA tiles for small ones, two kernels that run side by
// side on disjoint SMs and take tiles from two device-wide counters.
//
// "Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog", sections
// 2.1 and 7: under skewed routing one BM wastes either rows (large tiles on
// small experts) or bandwidth (small tiles on large experts), and BM should
// follow the expert sizes.  "Pearl's grouped GEMM kernel for MoE models,
// explained", "Four changes, three of them measured": 64-row tiles on a single
// CTA for small groups, the two-CTA mode for large ones.  A tcgen05 kernel
// uses one cta_group throughout, so the two tile shapes run as two kernels:
//
//   class P (m_e >= pair_min_rows): 256-row tiles on CTA pairs (the last tile
//     of an expert, when it holds <= 128 rows, as an M = 128 pair MMA);
//   class S (the other experts): 128-row tiles on one CTA (<= 64-row tails as
//     M = 64 MMAs).
//
// Each kernel builds both class lists from the device offsets (the routed
// counts never reach the host) and claims tiles of its own class first, in
// list order with each expert's tiles N tile by N tile, from a device counter
// (atomicAdd); when its class runs out it takes tiles of the other class: the
// pair kernel runs a class-S tile (<= 128 rows) as an M = 128 pair tile, the
// 1-CTA kernel runs a class-P tile as two 128-row tiles.  Every tile of both
// lists is claimed exactly once (the counter hands out each index once; an
// index past the end ends that class), so the result does not depend on how
// the SMs are split between the kernels or on whether they overlap at all.
// Claimed in list order, the tiles in flight at any moment are a contiguous
// window of the lists: the M tiles that read one weight panel run side by
// side, so the panel is read from HBM about once however the SMs drift.
//
// Without claims (GemmArgs::sched_claims = 0) each kernel walks its own
// class statically instead (ClassWalk), with no counters and no descriptor
// queue; a kernel whose partner has no CTAs walks the other class too, so the
// result never depends on how the SMs were split.
//
// The counters need no reset from the host between launches: sched[2]
// counts the CTAs of both kernels that have finished, and the last one
// (sched[2] reaching sched_total - 1) sets all three back to zero.  Every CTA
// takes part exactly once, on every exit path (a bounded wait that timed out
// and bad offsets included), after its last claim; a launch of the next call
// on the stream starts after both kernels end, so it finds the counters at
// zero.  (The host zeroes them once, with the handle's device word.)
#pragma once

#include <cstdint>

#include "rgg_tiles.cuh"

namespace rgg {

constexpr int kQueueDepth = 8;          // tile descriptors between a CTA's producer and its consumers
constexpr int kMixedBN = 256;           // both classes: MMAs 256 columns wide (plain: the last N tile narrowed;
                                        // fused gate-up: 128 gate + 128 up columns, 128 outputs)
constexpr int kPairMinRowsDefault = 256;

// The split of the SMs between the two kernels follows the estimated work of
// each class in SM-time, taken as the bytes each SM pulls into shared memory
// per tile (what set the pace of both tile shapes on a GB300): 2 (128 + c/2)
// for a 256-row pair tile of c columns (c rounded up to 128; 2 (64 + c/2) for
// a pair tile of <= 128 rows), 128 + c for a 128-row 1-CTA tile (c rounded up
// to 64; 64 + c for <= 64 rows), pair tiles weighted by 112/100: on the
// skewed 16k workload a pair tile's unit took 1.12 times a 1-CTA tile's
// (per-CTA traces), and the split this gives there (88 of 152 SMs on pairs)
// measured best.  Integer arithmetic, so the host planner (with the routed
// counts) and the kernels (from the device offsets) agree exactly.
struct MixedColCosts {
    int64_t p_full, p_half, s_full, s_half;  // per expert M tile, summed over its N tiles
};

__host__ __device__ inline MixedColCosts mixed_col_costs(int N) {
    MixedColCosts c = {0, 0, 0, 0};
    for (int c0 = 0; c0 < N; c0 += kMixedBN) {
        const int cols = (N - c0 < kMixedBN) ? N - c0 : kMixedBN;
        const int64_t pc = ((cols + 127) / 128) * 128;
        const int64_t sc = ((cols + 63) / 64) * 64;
        c.p_full += 2 * (128 + pc / 2);
        c.p_half += 2 * (64 + pc / 2);
        c.s_full += 128 + sc;
        c.s_half += 64 + sc;
    }
    return c;
}

// Adds expert rows m to the class costs.
__host__ __device__ inline void mixed_add_expert(const MixedColCosts& c, int64_t m, int pair_min_rows, int64_t* cost_p,
                                                 int64_t* cost_s) {
    if (m <= 0) return;
    if (m >= pair_min_rows) {
        const int64_t rem = m % 256;
        *cost_p += (m / 256) * c.p_full + (rem > 128 ? c.p_full : rem > 0 ? c.p_half : 0);
    } else {
        const int64_t rem = m % 128;
        *cost_s += (m / 128) * c.s_full + (rem > 64 ? c.s_full : rem > 0 ? c.s_half : 0);
    }
}

// SMs (even) for the pair kernel out of `sms`: all when there is no class-S
// work, none when there is no class-P work, else the cost share rounded up to
// an even count within [2, sms - 1].
__host__ __device__ inline int mixed_pair_sms(int64_t cost_p, int64_t cost_s, int sms) {
    if (cost_p <= 0) return 0;
    if (cost_s <= 0) return sms & ~1;
    const int64_t wp = 112 * cost_p, ws = 100 * cost_s;
    int pair = static_cast<int>((static_cast<int64_t>(sms) * wp + wp + ws) / (wp + ws)) & ~1;
    const int hi = (sms - 1) & ~1;
    pair = pair < 2 ? 2 : pair;
    return pair > hi ? hi : pair;
}

// The same split from the device offsets (one warp; lane 0 returns it).
__device__ __forceinline__ int mixed_pair_sms_from_offsets(const int32_t* s_off, int E, int N, int pair_min_rows,
                                                           int sms) {
    const int lane = threadIdx.x & 31;
    const MixedColCosts c = mixed_col_costs(N);
    int64_t cp = 0, cs = 0;
    for (int e = lane; e < E; e += 32) mixed_add_expert(c, s_off[e + 1] - s_off[e], pair_min_rows, &cp, &cs);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        cp += __shfl_xor_sync(0xffffffffu, cp, d);
        cs += __shfl_xor_sync(0xffffffffu, cs, d);
    }
    return mixed_pair_sms(cp, cs, sms);
}

struct ClassLists {
    const int32_t* s_off;
    const int32_t* s_preP;  // class P prefix of 256-row tiles
    const int32_t* s_preS;  // class S prefix of 128-row tiles
    int E, nN;
    int32_t nP, nS;
    int out_cols;           // output columns per tile: kMixedBN, or half of it for the fused gate-up op

    __device__ __forceinline__ TileCoord decode_p(int32_t t) const {
        return decode_tile(s_off, s_preP, E, 256, out_cols, nN, t, true);
    }
    __device__ __forceinline__ TileCoord decode_s(int32_t t) const {
        return decode_tile(s_off, s_preS, E, 128, out_cols, nN, t, true);
    }
};

// One CTA of a mixed launch is done with the counters (thread 0, once per
// CTA, after the CTA's last claim).
__device__ __forceinline__ void sched_cta_done(int32_t* sched, int32_t sched_total) {
    __threadfence();  // this CTA's claims before its count
    if (atomicAdd(sched + 2, 1) == sched_total - 1) {
        __threadfence();  // every other CTA's claims and counts before the reset
        atomicExch(sched + 0, 0);
        atomicExch(sched + 1, 0);
        atomicExch(sched + 2, 0);
    }
}

// Static walk over a kernel's share of the two classes (the launch without
// claims): positions [0, n_own) are the kernel's own class; when the other
// kernel has no CTAs, the other class follows (on the 1-CTA kernel each
// class-P tile as two positions, its two 128-row halves; an empty second half
// has rows <= 0 and is skipped by every role alike).  CTA or cluster k of a
// kernel of n takes positions k, k + n, ...
struct ClassWalk {
    bool pair_kernel;
    int32_t n_own, n_positions;

    __device__ __forceinline__ void init(const ClassLists& L, bool is_pair_kernel, bool other_kernel_has_ctas) {
        pair_kernel = is_pair_kernel;
        n_own = pair_kernel ? L.nP : L.nS;
        const int32_t other = other_kernel_has_ctas ? 0 : (pair_kernel ? L.nS : 2 * L.nP);
        n_positions = n_own + other;
    }

    __device__ __forceinline__ TileCoord at(const ClassLists& L, int32_t p) const {
        if (p < n_own) return pair_kernel ? L.decode_p(p) : L.decode_s(p);
        const int32_t q = p - n_own;
        if (pair_kernel) return L.decode_s(q);
        TileCoord c = L.decode_p(q >> 1);
        if (q & 1) {
            c.row0 += 128;
            c.rows -= 128;
        } else if (c.rows > 128) {
            c.rows = 128;
        }
        return c;
    }
};

__device__ __forceinline__ TileCoord sentinel_tile() {
    TileCoord c;
    c.expert = -1;
    c.row0 = 0;
    c.rows = 0;
    c.col0 = 0;
    return c;
}

// Claims of one CTA (the pair kernel: of the leader CTA).  The pair kernel
// claims class P first, the 1-CTA kernel class S first; `split_p` (the 1-CTA
// kernel) hands class-P tiles out as up to two 128-row tiles.  The first
// `off_p` tiles of class P belong to the pair kernel's clusters and the first
// `off_s` tiles of class S to the 1-CTA kernel's CTAs, one each, taken without
// an atomic (cluster or CTA k takes tile k of its own class), so no CTA waits
// for a counter before its first loads; claimed indices start after them.
// prefetch() issues the atomic of the next claim early so its latency hides
// under the current tile's loads; next() resolves it.
struct TileClaimer {
    int32_t* ctr_first;
    int32_t* ctr_second;
    int32_t n_first, n_second;
    int32_t off_first, off_second;
    bool first_is_p, split_p;
    int phase;          // 0: first class, 1: second class, 2: done
    int32_t own;        // this claimer's own first tile of its class, or -1 once taken
    bool has_half;      // the second 128-row half of a split class-P tile is due
    TileCoord half;
    bool ticket_valid;
    int32_t ticket;

    __device__ __forceinline__ void init(int32_t* sched, const ClassLists& L, bool pair_kernel, int32_t own_index,
                                         int32_t off_p, int32_t off_s) {
        first_is_p = pair_kernel;
        split_p = !pair_kernel;
        ctr_first = pair_kernel ? sched : sched + 1;
        ctr_second = pair_kernel ? sched + 1 : sched;
        n_first = pair_kernel ? L.nP : L.nS;
        n_second = pair_kernel ? L.nS : L.nP;
        off_first = pair_kernel ? off_p : off_s;
        off_second = pair_kernel ? off_s : off_p;
        phase = 0;
        own = own_index;
        has_half = false;
        ticket_valid = false;
        ticket = 0;
    }

    __device__ __forceinline__ int32_t claim() {
        return phase == 0 ? atomicAdd(ctr_first, 1) + off_first : atomicAdd(ctr_second, 1) + off_second;
    }

    __device__ __forceinline__ void prefetch() {
        ticket_valid = false;
        if (has_half || phase >= 2 || own >= 0) return;
        ticket = claim();
        ticket_valid = true;
    }

    __device__ __forceinline__ TileCoord next(const ClassLists& L) {
        if (has_half) {
            has_half = false;
            return half;
        }
        while (phase < 2) {
            int32_t t;
            if (own >= 0) {
                t = own;
                own = -1;
                if (t >= n_first) continue;  // no own tile: claim (indices past off_first)
            } else {
                t = ticket_valid ? ticket : claim();
                ticket_valid = false;
                if (t >= (phase == 0 ? n_first : n_second)) {
                    ++phase;
                    continue;
                }
            }
            const bool is_p = (phase == 0) == first_is_p;
            TileCoord c = is_p ? L.decode_p(t) : L.decode_s(t);
            if (is_p && split_p && c.rows > 128) {
                half = c;
                half.row0 = c.row0 + 128;
                half.rows = c.rows - 128;
                has_half = true;
                c.rows = 128;
            }
            return c;
        }
        return sentinel_tile();
    }
};

}  // namespace rgg
