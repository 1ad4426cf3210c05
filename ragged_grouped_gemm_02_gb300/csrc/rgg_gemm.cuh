// rgg_gemm.cuh -- the persistent, warp-specialized tcgen05 grouped GEMM kernel.
//
// Sources (by page title and section):
//  * "Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog":
//    section 2 (one flat, expert-major tile list; a tile owns its full K
//    reduction; partial tiles run the full MMA loop and mask their stores),
//    section 5 (TMA loads into a multistage shared-memory ring connected by
//    full/empty mbarriers with phase parity; 128-byte swizzle; a producer warp
//    separate from the math), section 7 (tcgen05: operands read from shared
//    memory through descriptors, the accumulator in TMEM, one thread issuing
//    the MMA for the CTA; BM chosen from the expert sizes).
//  * "Pearl's grouped GEMM kernel for MoE models, explained", "Four changes,
//    three of them measured": results go from registers straight to global
//    memory with 256-bit stores; 64-row tiles on a single CTA; the
//    accumulator's two halves are synchronised separately so one tile's
//    epilogue overlaps the next tile's main loop.
//
// CTA = 192 threads (320 for the fused gate-up and FP8 epilogues), one CTA per
// SM, persistent over tiles t = cta, cta+grid.. (or another walk order)
//   warp 0   : TMA producer (one lane)          smem ring  <- X tile, W tile
//   warp 1   : TMEM owner + MMA issuer (one lane) TMEM acc <- tcgen05.mma
//   warps 2-5: epilogue (2-9: two warps per      Y        <- TMEM via registers
//              TMEM lane quadrant, see epilogue_warps)
// The TMEM accumulator holds two BN-column buffers; acc_full/acc_empty
// barriers per buffer let the epilogue of tile i run under the MMAs of i+1.
//
// Operand layouts in shared memory (both written by TMA with 128B swizzle):
//   A (X rows, K-major): BM rows x 64 K = BM x 128 B per stage; 8-row groups
//     1024 B apart.  A K step of 16 elements is +32 B on the start address.
//   B (W, N-major = "MN-major"): BN/64 panels of 64 columns; a panel is 64 K
//     rows x 128 B (8 KiB).  LBO = panel stride (8 KiB), SBO = 1024 B (8 K rows).
//     A K step of 16 is +16 rows = +2048 B on the start address.
//
// Every wait is bounded by a global-timer limit.  On expiry the thread raises
// a CTA-wide abort flag and writes RGG_ERR_DEVICE_TIMEOUT to the status word;
// every role then leaves its loop, waits (again bounded) for its own
// in-flight copies or MMAs, and TMEM is freed before the CTA exits.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "rgg_checks.cuh"
#include "rgg_ptx.cuh"
#include "rgg_sched.cuh"
#include "rgg_tiles.cuh"

namespace rgg {

constexpr int kStatusTimeout = 5;
constexpr int kStatusBadOffsets = 4;
constexpr int kStatusBadRowIndex = 7;
constexpr int kStatusCapacity = 6;
constexpr int kMaxStages = 16;
// The CTA-pair kernel's static walk: the producer, which decodes every tile
// it loads, leaves the tile's MMA instruction descriptor for the MMA thread in
// a ring of kInfoSlots words in shared memory (slot = tile count mod
// kInfoSlots), written before its arrive on the tile's first stage; the MMA
// thread reads it after its wait on that stage (the arrive releases the
// write), so it runs no decode of its own between two tiles.  The producer is
// at most kMaxStages stages, so tiles, ahead: twice that many slots.
constexpr int kInfoSlots = 2 * kMaxStages;
constexpr int kThreads = 192;
constexpr int kBK = 64;                  // K elements per stage = one 128-byte swizzle row
constexpr uint64_t kDrainLimitNs = 2000000000ull;  // teardown waits for copies/MMAs already issued
constexpr int32_t kDebugProducerStall = 1;  // test hook: the producer issues nothing

struct GemmArgs {
    const int32_t* offsets;  // device int32 [E+1]
    __nv_bfloat16* Y;        // device bf16 [M_tot, N]
    int32_t* status;         // device status word
    int64_t M_tot;
    int32_t E, K, N;
    int32_t num_k_blocks;    // ceil(K / 64)
    int32_t n_tiles_n;       // ceil(N / BN)
    int32_t stages;
    int32_t y_vec32;         // 1: rows of Y are 32-byte aligned (256-bit stores)
    int32_t debug_flags;     // 0 in normal use; kDebugProducerStall for failure-detection tests
    int32_t tail64;          // 1: tiles holding <= 64 rows run as 64-row MMAs (128-row kernels)
    int32_t walk_order = 0;  // order of the persistent walk over the tile list (rgg_tiles.cuh)
    uint64_t timeout_ns;
    const float* sx = nullptr;  // FP8 kernels: fp32 scale of each row of X [M_tot]
    const float* sw = nullptr;  // FP8 kernels: fp32 scale of each (expert, column) of W [E, N]
    const int32_t* row_index = nullptr;  // gather kernels: token row of each routed row [M_tot]
    int32_t t_rows = 0;                  // gather kernels: rows of the token matrix
    // Mixed launch (rgg_sched.cuh): tiles claimed from two device counters
    // sched[0] (class P) and sched[1] (class S); sched[2] counts finished CTAs
    // of the sched_total CTAs of both kernels (the last one resets all three).
    int32_t* sched = nullptr;
    int32_t sched_total = 0;
    int32_t sched_pairs = 0;    // clusters of the pair kernel (each takes its first class-P tile without a claim)
    int32_t sched_singles = 0;  // CTAs of the 1-CTA kernel (each takes its first class-S tile without a claim)
    int32_t sched_claims = 1;   // 0: each kernel walks its own class statically (no counters, no queue)
    int32_t pair_min_rows = kPairMinRowsDefault;
    // Fixed walks only.  1: both kernels were launched over all split_sms
    // SMs (the pair kernel on split_sms & ~1 of them); each CTA computes the
    // split from the device offsets (mixed_pair_sms_from_offsets) and the
    // clusters and CTAs past their kernel's share leave at once.  0: the
    // launched grids are the split.
    int32_t sched_split = 0;
    int32_t split_sms = 0;
    // 1: the kernel waits for the grid before it on the stream before its
    // first global memory access (programmatic dependent launch, see
    // pdl_wait_prerequisites); 0 only for the mixed launch's 1-CTA kernel
    // beside a pair kernel, which waits at its end instead.
    int32_t pdl_wait_first = 1;
};

// Shared-memory carve-up shared by the host planner and the kernel.  Offsets
// are from a 1024-byte aligned base; the host adds 1024 bytes of slack for
// aligning the dynamic shared-memory window.
struct SmemPlan {
    uint32_t a_stage, b_stage, a_off, b_off, bar_off, misc_off, off_off, pre_off, ord_off, spre_off, q_off,
        qbar_off, total;
};

// `sorted`: room for the size-sorted walk (expert order and its tile
// prefix).  `mixed`: room for the second class prefix (at ord_off) and the
// tile queue (kQueueDepth 16-byte descriptors, then q_full[Q], q_empty[Q]).
__host__ __device__ inline SmemPlan smem_plan(int BM, int BN, int stages, int E, bool sorted = false,
                                              bool mixed = false) {
    SmemPlan p;
    const uint32_t ex = 4u * static_cast<uint32_t>(E + 1);
    p.a_stage = static_cast<uint32_t>(BM) * 128u;
    p.b_stage = static_cast<uint32_t>(BN) * 128u;
    p.a_off = 0;
    p.b_off = p.a_off + stages * p.a_stage;
    p.bar_off = p.b_off + stages * p.b_stage;          // full[S], empty[S], acc_full[2], acc_empty[2], drain
    // misc: tmem base, abort flag, the mixed launch's SM split, one spare word,
    // then the pair kernel's ring of kInfoSlots instruction descriptors
    p.misc_off = p.bar_off + 8u * (2u * stages + 5u);
    p.off_off = p.misc_off + 16u + 4u * kInfoSlots;
    p.pre_off = p.off_off + ex;
    p.ord_off = p.pre_off + ex;
    p.spre_off = p.ord_off + ((sorted || mixed) ? ex : 0u);
    p.q_off = (p.spre_off + (sorted ? ex : 0u) + 15u) & ~15u;
    p.qbar_off = p.q_off + (mixed ? 16u * kQueueDepth : 0u);
    p.total = p.qbar_off + (mixed ? 16u * kQueueDepth : 0u);
    return p;
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              int32_t* status, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            atomicCAS(status, 0, kStatusTimeout);
            return false;
        }
    }
}

// Used only while tearing down after an abort: waits for the barrier without
// looking at the abort flag, still bounded by the time limit.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > timeout_ns) return false;
    return true;
}

// Kernels on clusters of two CTAs: as wait_or_abort, and a timeout also raises
// the other CTA's abort flag (its shared::cluster address), so both leave
// their loops instead of waiting on arrivals that will not come.
// kClusterAcquire: the barrier is arrived on by the other CTA after it wrote
// (or read) this CTA's shared memory, so the wait acquires at cluster scope.
template <bool kClusterAcquire = false>
__device__ __forceinline__ bool pair_wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                   uint32_t peer_flag_cluster, int32_t* status, uint64_t timeout_ns) {
    auto probe = [&]() { return kClusterAcquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (probe()) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (probe()) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            st_shared_cluster_u32(peer_flag_cluster, 1u);
            atomicCAS(status, 0, kStatusTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

// Element traits.  Every stage row is one 128-byte swizzle row, so a bf16
// stage covers K = 64 and an FP8 (E4M3) stage K = 128, with the same bytes:
// A is BM x 128 B, B is BN/kPanelN panels of kKStage K rows x 128 B.
template <int BM, int BN, bool kFp8 = false>
struct TileConfig {
    static_assert(BM == 64 || BM == 128, "tcgen05 cta_group::1 tiles are 64 or 128 rows");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN is a multiple of one 64-column panel, at most 256");
    static_assert(!kFp8 || BN % 128 == 0, "FP8 weight panels are 128 columns wide");
    static constexpr int kKStage = kFp8 ? 128 : 64;                        // K elements per stage
    static constexpr int kPanelN = kFp8 ? 128 : 64;                        // W columns per panel
    static constexpr uint32_t kPanelB = static_cast<uint32_t>(kKStage) * 128u;  // bytes per W panel
    static constexpr uint32_t kBStep = kFp8 ? 4096u : 2048u;  // B start advance per MMA (32 or 16 K rows)
    static constexpr uint32_t kTmemCols = (2 * BN <= 256) ? 256u : 512u;  // two accumulator buffers
    // Instruction descriptor for an M x n MMA (n = the panels a tile loads x kPanelN).
    __host__ __device__ static constexpr uint32_t idesc(int m, int n) {
        return kFp8 ? idesc_e4m3_f32(m, n, true) : idesc_bf16_f32(m, n, true);
    }
};


constexpr int kMmasPerStage = 4;  // K = 16 (bf16) or 32 (FP8) per instruction

// A 128-row tile whose rows are the last <= 64 of its expert runs as a
// 64-row MMA (the "tail64" mode): the tile list is unchanged, only the MMA
// height, the X box and the epilogue's TMEM lane mapping follow the tile.
template <int BM>
__device__ __forceinline__ bool runs_as_64_rows(const GemmArgs& args, const TileCoord& c) {
    return BM == 64 || (args.tail64 != 0 && c.rows <= 64);
}

// Epilogue modes.  kEpiPlain stores the accumulator.  kEpiSwiGLU is the fused
// gate-up projection: W holds 2N columns (gate [0, N), up [N, 2N)); a tile of
// BN/2 output columns loads the matching BN/2 gate and BN/2 up columns into one
// B stage, one MMA of width BN puts gate | up side by side in TMEM, and the
// epilogue writes silu(gate) * up.
constexpr int kEpiPlain = 0;
constexpr int kEpiSwiGLU = 1;

// Weight panels a tile loads and multiplies.  A plain tile whose columns run
// past N (the last N tile of an expert) loads only the panels that hold
// columns below N and issues an MMA of that width, so neither the copies nor
// the MMAs of the columns past N are paid for (on N = 2688 with 256-column
// tiles every expert's eleventh N tile is half empty).  The fused gate-up
// tile keeps its gate | up panel layout and loads them all.
template <int kPanels, int kPanelN, int kEpi>
__device__ __forceinline__ int tile_panels(int32_t col0, int32_t N) {
    if (kEpi != kEpiPlain) return kPanels;
    const int32_t need = (N - col0 + kPanelN - 1) / kPanelN;
    return need < kPanels ? static_cast<int>(need) : kPanels;
}

// Epilogue warps of the 1-CTA kernel.  Four (one per TMEM lane quadrant)
// keep pace with the main loop for plain bf16 outputs.  The FP8 epilogue also
// loads and applies the row and column scales, and the fused gate-up epilogue
// reads two accumulator halves and evaluates an exponential per output; with
// four warps both outlasted short main loops (K = 1024: the MMA waited on the
// accumulator), so they run two warps per quadrant, each on half of the tile's
// columns.  Measured on a GB300: FP8 uniform 975 -> 1 370 TFLOP/s, fused
// gate-up uniform 914 -> 1 000 and skew16k 696 -> 816; for plain bf16 the
// same split lost 3-5 %.
template <int kEpi, bool kFp8>
__host__ __device__ constexpr int epilogue_warps() {
    return (kFp8 || kEpi == kEpiSwiGLU) ? 8 : 4;
}
template <int kEpi, bool kFp8>
__host__ __device__ constexpr int cta_threads() {
    return 64 + 32 * epilogue_warps<kEpi, kFp8>();
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + __expf(-z)); }

// Epilogue of one finished accumulator buffer of a 1-CTA tile, for one
// epilogue warp: lane `lane` of the warp holds tile row r_local (TMEM row
// address t_row: the warp's lane quadrant and the buffer's first column) and
// writes columns [cc0, cc0 + kOutN / parts) of it, 32 at a time, through
// registers to Y with 256-bit stores ("Pearl's grouped GEMM kernel for MoE
// models, explained").  Rows past the tile's valid rows, and every row when
// `store` is false, are read from TMEM but not written.
//
// [row_lo, row_hi) are the expert's rows and tcol the buffer's first TMEM
// column, read only by the bounds checks of the debug build.
template <int BN, int kEpi, bool kFp8>
__device__ __forceinline__ void epilogue_store_tile(const GemmArgs& args, const TileCoord& c, bool half, int r_local,
                                                    uint32_t t_row, int lane, int cc0, bool store, int32_t row_lo,
                                                    int32_t row_hi, uint32_t tcol) {
    constexpr int kOutN = (kEpi == kEpiSwiGLU) ? BN / 2 : BN;
    constexpr int kPartCols = kOutN / (epilogue_warps<kEpi, kFp8>() / 4);
    constexpr uint32_t kTmemCols = TileConfig<64, BN, kFp8>::kTmemCols;
    const int N = args.N;
    const bool row_ok = store && (!half || lane < 16) && (r_local < c.rows);
    const int64_t row = static_cast<int64_t>(c.row0) + r_local;
    __nv_bfloat16* yrow = args.Y + row * N + c.col0;
#pragma unroll 1
    for (int cc = cc0; cc < cc0 + kPartCols; cc += 32) {
        if (c.col0 + cc >= N) break;  // columns past N: not computed (tile_panels), not stored
        uint32_t v[32];
        const bool ld_ok = RGG_BOUNDS_OK(tmem_cols_ok(tcol + cc, 32, kTmemCols), args.status);
        if (ld_ok) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(cc), v);
        if (kEpi == kEpiSwiGLU) {
            // gate in columns [cc, cc+32), up in [kOutN + cc, kOutN + cc + 32)
            uint32_t u[32];
            const bool ldu_ok = RGG_BOUNDS_OK(tmem_cols_ok(tcol + kOutN + cc, 32, kTmemCols), args.status);
            if (ldu_ok) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(kOutN + cc), u);
            tmem_ld_wait();
            if (!ldu_ok)
                for (int i = 0; i < 32; ++i) u[i] = 0u;
            if (!ld_ok)
                for (int i = 0; i < 32; ++i) v[i] = 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[i] = __float_as_uint(silu_f32(__uint_as_float(v[i])) * __uint_as_float(u[i]));
        } else {
            tmem_ld_wait();
            if (!ld_ok)
                for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if constexpr (kFp8) {
            // dequantise: row scale of X times the expert's column scale of W
            if (row_ok && RGG_BOUNDS_OK(store_ok(row, c.col0 + cc, 0, row_lo, row_hi, N) && c.col0 + cc + 16 <= N,
                                        args.status)) {
                const float rs = __ldg(args.sx + c.row0 + r_local);
                const float* swp = args.sw + static_cast<int64_t>(c.expert) * N + c.col0 + cc;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (c.col0 + cc + 16 * h < N) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float4 s4 = __ldg(reinterpret_cast<const float4*>(swp + 16 * h) + q4);
                            const int i0 = 16 * h + 4 * q4;
                            v[i0 + 0] = __float_as_uint(__uint_as_float(v[i0 + 0]) * rs * s4.x);
                            v[i0 + 1] = __float_as_uint(__uint_as_float(v[i0 + 1]) * rs * s4.y);
                            v[i0 + 2] = __float_as_uint(__uint_as_float(v[i0 + 2]) * rs * s4.z);
                            v[i0 + 3] = __float_as_uint(__uint_as_float(v[i0 + 3]) * rs * s4.w);
                        }
                    }
                }
            }
        }
        if (row_ok) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = c.col0 + cc + 16 * h;
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[16 * h + 2 * i], v[16 * h + 2 * i + 1]);
                __nv_bfloat16* dst = yrow + cc + 16 * h;
                if (col + 16 <= N) {
                    if (RGG_BOUNDS_OK(store_ok(row, col, 16, row_lo, row_hi, N), args.status)) {
                        if (args.y_vec32) {
                            st_global_v8(dst, w);
                        } else {
                            st_global_v4(dst, w[0], w[1], w[2], w[3]);
                            st_global_v4(dst + 8, w[4], w[5], w[6], w[7]);
                        }
                    }
                } else if (col + 8 <= N) {
                    if (RGG_BOUNDS_OK(store_ok(row, col, 8, row_lo, row_hi, N), args.status))
                        st_global_v4(dst, w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
}

// Token gather fused into the A loads (kGatherTma): the A rows are gathered
// from a token matrix X_tok [T, K] through args.row_index (routed row i
// reads token row_index[i]); tmap_x is the token matrix with a one-row box
// and tmap_x64 is unused.  The producer warp loads four rows per TMA
// tile::gather4 copy, one lane per group of four tile rows, and copies only
// the groups that hold rows of the tile's expert.  Each gathered row is a
// separate 128-byte fetch, and an A tile is fetched again for every N tile,
// so this suits tiles of few rows (small expert groups); large groups are
// gathered once by gather_rows_kernel and multiplied by the plain kernel.
constexpr int kGatherNone = 0;
constexpr int kGatherTma = 1;

// kDyn: the 1-CTA kernel of the mixed launch (rgg_sched.cuh).  Its producer
// claims tiles from the device counters and hands each tile's descriptor to
// the MMA thread and the epilogue warps through a small shared-memory queue
// (q_full / q_empty barriers per slot); a descriptor with expert -1 ends the
// walk.  Otherwise each role decodes the static walk t = cta, cta + grid, ...
template <int BM, int BN, int kEpi = kEpiPlain, bool kFp8 = false, int kGather = kGatherNone, bool kDyn = false>
__global__ void __launch_bounds__(cta_threads<kEpi, kFp8>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_x64,
                        const __grid_constant__ CUtensorMap tmap_w, const GemmArgs args) {
    using Cfg = TileConfig<BM, BN, kFp8>;
    static_assert(!kDyn || (BM == 128 && BN == kMixedBN && !kFp8 && kGather == kGatherNone),
                  "the mixed launch's 1-CTA kernel runs bf16 128 x 256 tiles (plain or fused gate-up)");
    static_assert(kEpi == kEpiPlain || (BN % 128) == 0, "fused gate-up tiles hold whole gate and up panels");
    static_assert(!(kFp8 && kEpi == kEpiSwiGLU), "the fused gate-up epilogue is bf16 only");
    static_assert(!(kFp8 && kGather != kGatherNone), "the token gather is bf16 only");
    static_assert(BM / 4 <= 32, "one producer lane per group of four tile rows");
    constexpr int kOutN = (kEpi == kEpiSwiGLU) ? BN / 2 : BN;  // output columns per tile
    constexpr int kPanels = BN / Cfg::kPanelN;
    constexpr int kElemBytes = kFp8 ? 1 : 2;
    const int64_t kNw = (kEpi == kEpiSwiGLU) ? 2 * static_cast<int64_t>(args.N) : args.N;  // columns of W
    (void)kNw;
    // A plain tile loads only panels below N (tile_panels); the fused gate-up
    // tile's last up panel of an expert's last N tile can start past column
    // 2N, a box the copy zero-fills.
    constexpr int64_t kWOverhang = (kEpi == kEpiSwiGLU) ? Cfg::kPanelN : 0;
    // Column of W read by B panel p of a tile whose first output column is col0.
    auto w_col = [&](int32_t col0, int p) -> int32_t {
        if (kEpi == kEpiSwiGLU)
            return (p < kPanels / 2) ? col0 + Cfg::kPanelN * p : args.N + col0 + Cfg::kPanelN * (p - kPanels / 2);
        return col0 + Cfg::kPanelN * p;
    };
    extern __shared__ __align__(1024) uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = args.E;
    const int S = args.stages;

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const SmemPlan sp = smem_plan(BM, BN, S, E, !kDyn && args.walk_order == 3, kDyn);
    const uint32_t a0 = base + sp.a_off;
    const uint32_t b0 = base + sp.b_off;
    const uint32_t bars = base + sp.bar_off;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + sp.misc_off);
    int32_t* s_off = reinterpret_cast<int32_t*>(gbase + sp.off_off);
    int32_t* s_pre = reinterpret_cast<int32_t*>(gbase + sp.pre_off);
    int32_t* s_order = reinterpret_cast<int32_t*>(gbase + sp.ord_off);  // walk order 3; mixed: class S prefix
    int32_t* s_spre = reinterpret_cast<int32_t*>(gbase + sp.spre_off);
    int32_t* q_desc = reinterpret_cast<int32_t*>(gbase + sp.q_off);     // mixed: tile queue
    auto qfull_bar = [&](int i) { return base + sp.qbar_off + 8u * i; };
    auto qempty_bar = [&](int i) { return base + sp.qbar_off + 8u * (kQueueDepth + i); };

    // Launched with programmatic stream serialisation: the grid may be
    // resident before the kernel ahead of it on the stream has finished, so
    // it touches no global memory before that kernel's writes are visible.
    // Then the grid after it may launch; its CTAs take the SMs this grid's
    // CTAs leave and wait the same way.
    if (args.pdl_wait_first) pdl_wait_prerequisites();
    pdl_launch_dependents();

    // S1: group offsets -> validated per-expert tile prefix.
    if (!load_and_check_offsets(args.offsets, s_off, E, args.M_tot)) {
        if (threadIdx.x == 0) atomicCAS(args.status, 0, kStatusBadOffsets);
        if constexpr (kDyn) {
            if (threadIdx.x == 0 && args.sched_claims) sched_cta_done(args.sched, args.sched_total);
            pdl_wait_prerequisites();
        }
        return;
    }
    ClassLists L;
    int32_t T;
    // mixed launch, fixed walks: clusters of the pair kernel and CTAs of this
    // kernel that take part (this kernel's CTA k walks positions k, k + units, ...)
    int32_t pair_units = 0, single_units = 0;
    if constexpr (kDyn) {
        // both class lists (class P in s_pre, class S in s_order)
        if (warp == 0) build_class_prefix_warp(s_off, s_pre, E, 256, args.n_tiles_n, args.pair_min_rows, 0x7fffffff);
        if (warp == 1) build_class_prefix_warp(s_off, s_order, E, 128, args.n_tiles_n, 0, args.pair_min_rows);
        if (warp == 2 && args.sched_split) {
            const int ps = mixed_pair_sms_from_offsets(s_off, E, kEpi == kEpiSwiGLU ? 2 * args.N : args.N,
                                                       args.pair_min_rows, args.split_sms);
            if (lane == 0) misc[2] = static_cast<uint32_t>(ps);
        }
        __syncthreads();
        L = ClassLists{s_off, s_pre, s_order, E, args.n_tiles_n, s_pre[E], s_order[E], kOutN};
        T = L.nP + L.nS;
        if (T == 0) {
            if (threadIdx.x == 0 && args.sched_claims) sched_cta_done(args.sched, args.sched_total);
            pdl_wait_prerequisites();
            return;
        }
        pair_units = args.sched_split ? static_cast<int32_t>(misc[2]) / 2 : args.sched_pairs;
        single_units = args.sched_split ? args.split_sms - static_cast<int32_t>(misc[2]) : args.sched_singles;
        if (args.sched_split && static_cast<int32_t>(blockIdx.x) >= single_units) {
            // past this kernel's share: leave (CTA 0 still keeps the grid from
            // ending before the pair kernel)
            if (blockIdx.x == 0) pdl_wait_prerequisites();
            return;
        }
    } else {
        if (warp == 0) build_tile_prefix_warp(s_off, s_pre, E, BM, args.n_tiles_n);
        __syncthreads();
        T = s_pre[E];
        if (args.walk_order == 3) build_size_order(s_off, s_order, s_spre, E, BM, args.n_tiles_n);
        if (static_cast<int32_t>(blockIdx.x) >= T) return;  // uniform over the CTA
    }

    if (threadIdx.x == 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), epilogue_warps<kEpi, kFp8>());
        }
        mbar_init(drain_bar, 1);
        if constexpr (kDyn) {
            for (int i = 0; i < kQueueDepth; ++i) {
                mbar_init(qfull_bar(i), 1);
                mbar_init(qempty_bar(i), 1 + epilogue_warps<kEpi, kFp8>());
            }
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmap_x);
        tma_prefetch_map(&tmap_x64);
        tma_prefetch_map(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&misc[0]), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const uint32_t tmem_base = misc[0];
    volatile uint32_t* abort_flag = &misc[1];
    const int KB = args.num_k_blocks;
    const int nN = args.n_tiles_n;
    const int WO = args.walk_order;  // walk position t visits tile walk_tile(t, ...)
    const int32_t WS = walk_stride_for(T);
    // The tile visited at walk position p.
    auto tile_at = [&](int32_t p) -> TileCoord {
        return walk_decode(s_off, s_pre, s_order, s_spre, E, BM, kOutN, nN, T, WO, WS, p);
    };
    // Mixed launch: a consumer takes the next descriptor from the queue
    // (`warp_wide`: all lanes of an epilogue warp wait, lane 0 releases the
    // slot for the warp).  False on an abort; expert -1 ends the walk.
    auto q_pop = [&](int& qs, uint32_t& qp, TileCoord& c, bool warp_wide) -> bool {
        bool ok = wait_or_abort(qfull_bar(qs), qp, abort_flag, args.status, args.timeout_ns);
        if (warp_wide) ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        const volatile int32_t* d = q_desc + 4 * qs;
        c.expert = d[0];
        c.row0 = d[1];
        c.rows = d[2];
        c.col0 = d[3];
        if (warp_wide) {
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty_bar(qs));
        } else {
            mbar_arrive(qempty_bar(qs));
        }
        if (++qs == kQueueDepth) {
            qs = 0;
            qp ^= 1u;
        }
        return true;
    };

    if (kGather == kGatherTma && warp == 0) {
        // ------------------------------------- S4 with the token gather (TMA)
        // Lane l owns tile rows 4l..4l+3.  The token indices of the next
        // tile are loaded while the current tile's stages are issued, so
        // their latency stays off the ring.  A row past the tile's last row
        // in a partly filled group repeats the group's first row (its product
        // is never stored); an index outside [0, T) is reported and replaced
        // by token 0, so every copy stays inside the token matrix.
        if ((args.debug_flags & kDebugProducerStall) == 0) {
            int st = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = true;
            int32_t nxt[4] = {0, 0, 0, 0};
            TileCoord cn = {0, 0, 0, 0};
            auto fetch = [&](int32_t p) {
                cn = tile_at(p);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * lane + i < cn.rows ? 4 * lane + i : 4 * lane;
                    nxt[i] = (4 * lane < cn.rows) ? __ldg(args.row_index + cn.row0 + r) : 0;
                }
            };
            if (static_cast<int32_t>(blockIdx.x) < T) fetch(blockIdx.x);
            for (int32_t t = blockIdx.x; ok && t < T; t += gridDim.x) {
                const TileCoord c = cn;
                int32_t tok[4];
                bool bad = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    tok[i] = nxt[i];
                    if (tok[i] < 0 || tok[i] >= args.t_rows) {
                        bad = true;
                        tok[i] = 0;
                    }
                }
                const int groups = (c.rows + 3) >> 2;
                if (bad && 4 * lane < c.rows) atomicCAS(args.status, 0, kStatusBadRowIndex);
                if (t + static_cast<int32_t>(gridDim.x) < T) fetch(t + gridDim.x);
                const int np = tile_panels<kPanels, Cfg::kPanelN, kEpi>(c.col0, args.N);
                const uint32_t tx_bytes = static_cast<uint32_t>(groups) * 512u + np * Cfg::kPanelB;
                for (int kb = 0; kb < KB; ++kb) {
                    int got = 1;
                    if (lane == 0) got = wait_or_abort(empty_bar(st), ph ^ 1u, abort_flag, args.status, args.timeout_ns);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(full_bar(st), tx_bytes);
                    __syncwarp();
                    if (lane < groups &&
                        RGG_BOUNDS_OK(x_box_ok(kb * Cfg::kKStage, tok[0], args.K, args.t_rows, kElemBytes) &&
                                          x_box_ok(kb * Cfg::kKStage, tok[3], args.K, args.t_rows, kElemBytes),
                                      args.status))
                        tma_gather4(a0 + st * sp.a_stage + 512u * lane, &tmap_x, full_bar(st), kb * Cfg::kKStage,
                                    tok[0], tok[1], tok[2], tok[3]);
                    if (lane == 0) {
#pragma unroll
                        for (int p = 0; p < kPanels; ++p)
                            if (p < np && RGG_BOUNDS_OK(w_box_ok(w_col(c.col0, p), kb * Cfg::kKStage, c.expert, kNw,
                                                                 args.K, E, kElemBytes, kWOverhang),
                                                        args.status))
                                tma_load_3d(b0 + st * sp.b_stage + p * Cfg::kPanelB, &tmap_w, full_bar(st),
                                            w_col(c.col0, p), kb * Cfg::kKStage, c.expert);
                    }
                    ++issued;
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && lane == 0) {
                // Let the copies already issued land before the CTA can exit.
                const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
                for (uint32_t i = issued - n; i < issued; ++i)
                    wait_bounded(full_bar(static_cast<int>(i % S)), (i / S) & 1u, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------------------------------------------- S4: TMA producer
        if (lane == 0 && (args.debug_flags & kDebugProducerStall) == 0) {
            int st = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = true;
            auto produce = [&](const TileCoord& c) {
                (void)RGG_BOUNDS_OK(tile_ok(c.expert, c.row0, c.rows, c.col0, s_off, E, args.N), args.status);
                const bool half = runs_as_64_rows<BM>(args, c);
                const int np = tile_panels<kPanels, Cfg::kPanelN, kEpi>(c.col0, args.N);
                const uint32_t tx_bytes = (half ? 64u : static_cast<uint32_t>(BM)) * 128u + np * Cfg::kPanelB;
                const CUtensorMap* xmap = (BM == 128 && half) ? &tmap_x64 : &tmap_x;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_or_abort(empty_bar(st), ph ^ 1u, abort_flag, args.status, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(st), tx_bytes);
                    if (RGG_BOUNDS_OK(x_box_ok(kb * Cfg::kKStage, c.row0, args.K, args.M_tot, kElemBytes),
                                      args.status))
                        tma_load_2d(a0 + st * sp.a_stage, xmap, full_bar(st), kb * Cfg::kKStage, c.row0);
#pragma unroll
                    for (int p = 0; p < kPanels; ++p)
                        if (p < np && RGG_BOUNDS_OK(w_box_ok(w_col(c.col0, p), kb * Cfg::kKStage, c.expert, kNw,
                                                             args.K, E, kElemBytes, kWOverhang),
                                                    args.status))
                            tma_load_3d(b0 + st * sp.b_stage + p * Cfg::kPanelB, &tmap_w, full_bar(st),
                                        w_col(c.col0, p), kb * Cfg::kKStage, c.expert);
                    ++issued;
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            };
            if (kDyn && !args.sched_claims) {
                ClassWalk cw;
                cw.init(L, false, pair_units > 0);
                for (int32_t p = blockIdx.x; ok && p < cw.n_positions; p += single_units) {
                    const TileCoord c = cw.at(L, p);
                    if (c.rows > 0) produce(c);
                }
            } else if constexpr (kDyn) {
                // claim, hand the descriptor to the consumers, load the tile
                TileClaimer cl;
                cl.init(args.sched, L, false, blockIdx.x, args.sched_pairs, args.sched_singles);
                int qs = 0;
                uint32_t qp = 0;
                TileCoord c = cl.next(L);
                while (ok) {
                    if (!wait_or_abort(qempty_bar(qs), qp ^ 1u, abort_flag, args.status, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    int32_t* d = q_desc + 4 * qs;
                    d[0] = c.expert;
                    d[1] = c.row0;
                    d[2] = c.rows;
                    d[3] = c.col0;
                    mbar_arrive(qfull_bar(qs));
                    if (++qs == kQueueDepth) {
                        qs = 0;
                        qp ^= 1u;
                    }
                    if (c.expert < 0) break;
                    cl.prefetch();
                    produce(c);
                    if (ok) c = cl.next(L);
                }
            } else {
                for (int32_t t = blockIdx.x; ok && t < T; t += gridDim.x) produce(tile_at(t));
            }
            if (!ok) {
                // Let the copies already issued land before the CTA can exit.
                const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
                for (uint32_t i = issued - n; i < issued; ++i)
                    wait_bounded(full_bar(static_cast<int>(i % S)), (i / S) & 1u, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ S5: MMA issuer
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true;
            auto mma_tile = [&](const TileCoord& c) {
                const int np = tile_panels<kPanels, Cfg::kPanelN, kEpi>(c.col0, args.N);
                const uint32_t idesc = Cfg::idesc(runs_as_64_rows<BM>(args, c) ? 64 : BM, np * Cfg::kPanelN);
                if (!wait_or_abort(acce_bar(acc), acc_ph ^ 1u, abort_flag, args.status, args.timeout_ns)) {
                    ok = false;
                    return;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_or_abort(full_bar(st), ph, abort_flag, args.status, args.timeout_ns)) {
                        ok = false;
                        return;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_st = a0 + st * sp.a_stage;
                    const uint32_t b_st = b0 + st * sp.b_stage;
#pragma unroll
                    for (int j = 0; j < kMmasPerStage; ++j) {
                        const uint64_t ad = sw128_desc(a_st + 32u * j, 16u, 1024u);
                        const uint64_t bd = sw128_desc(b_st + Cfg::kBStep * j, Cfg::kPanelB, 1024u);
                        if constexpr (kFp8)
                            mma_f8_ss(d_tmem, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
                        else
                            mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(st));  // frees the stage once these MMAs have read it
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit(accf_bar(acc));      // accumulator buffer ready for the epilogue
                if (++acc == 2) {
                    acc = 0;
                    acc_ph ^= 1u;
                }
            };
            if (kDyn && !args.sched_claims) {
                ClassWalk cw;
                cw.init(L, false, pair_units > 0);
                for (int32_t p = blockIdx.x; ok && p < cw.n_positions; p += single_units) {
                    const TileCoord c = cw.at(L, p);
                    if (c.rows > 0) mma_tile(c);
                }
            } else if constexpr (kDyn) {
                int qs = 0;
                uint32_t qp = 0;
                TileCoord c;
                while (ok) {
                    if (!q_pop(qs, qp, c, false)) {
                        ok = false;
                        break;
                    }
                    if (c.expert < 0) break;
                    mma_tile(c);
                }
            } else {
                for (int32_t t = blockIdx.x; ok && t < T; t += gridDim.x) mma_tile(tile_at(t));
            }
            if (!ok) {
                mma_commit(drain_bar);
                wait_bounded(drain_bar, 0u, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- S6: epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        constexpr int kParts = epilogue_warps<kEpi, kFp8>() / 4;  // warps per quadrant
        constexpr int kPartCols = kOutN / kParts;                  // tile columns each of them writes
        static_assert(kPartCols % 32 == 0, "each epilogue warp handles whole 32-column chunks");
        const int cc0 = ((warp - 2) >> 2) * kPartCols;
        int acc = 0;
        uint32_t acc_ph = 0;
        // false when the CTA aborts
        auto epi_tile = [&](const TileCoord& c) -> bool {
            // M = 128: tile row 32q + lane sits in TMEM lane 32q + lane.  M = 64:
            // tile row 16q + i sits in TMEM lane 32q + i (i < 16).
            const bool half = runs_as_64_rows<BM>(args, c);
            const int r_local = half ? (q * 16 + (lane & 15)) : (q * 32 + lane);
            bool ok = wait_or_abort(accf_bar(acc), acc_ph, abort_flag, args.status, args.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) return false;
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            epilogue_store_tile<BN, kEpi, kFp8>(args, c, half, r_local, t_row, lane, cc0, true, s_off[c.expert],
                                                s_off[c.expert + 1], static_cast<uint32_t>(acc * BN));
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1u;
            }
            return true;
        };
        if (kDyn && !args.sched_claims) {
            ClassWalk cw;
            cw.init(L, false, pair_units > 0);
            for (int32_t p = blockIdx.x; p < cw.n_positions; p += single_units) {
                const TileCoord c = cw.at(L, p);
                if (c.rows > 0 && !epi_tile(c)) break;
            }
        } else if constexpr (kDyn) {
            int qs = 0;
            uint32_t qp = 0;
            TileCoord c;
            while (q_pop(qs, qp, c, true) && c.expert >= 0)
                if (!epi_tile(c)) break;
        } else {
            for (int32_t t = blockIdx.x; t < T; t += gridDim.x)
                if (!epi_tile(tile_at(t))) break;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
    // The mixed launch's 1-CTA kernel may start before the pair kernel ends;
    // it does not end before it, so the stream's later work sees both done.
    if constexpr (kDyn) {
        if (threadIdx.x == 0 && args.sched_claims) sched_cta_done(args.sched, args.sched_total);  // after the producer's last claim
        pdl_wait_prerequisites();
    }
}

}  // namespace rgg
