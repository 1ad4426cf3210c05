// rgg_api.cu -- the C ABI of librgg.so (declared in include/rgg.h): argument
// checks, the tile-shape planner, TMA descriptor encoding and the launches.
//
// The planner follows "Grouped GEMM for Imbalanced Experts on Blackwell: A
// WIP Worklog", section 6 ("BM therefore has to be selected from both the
// expert sizes and the rate each tile shape achieves") and section 7 (choose
// BM from the expert-size distribution), and "Pearl's grouped GEMM kernel for
// MoE models, explained", "Four changes, three of them measured" (64-row
// tiles where experts average 64 rows or fewer).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "rgg.h"
#include "rgg_internal.h"

struct rgg_handle {
    int device;
    int num_sms;
    int smem_optin;
    int32_t* d_status;
};

namespace {

thread_local std::string g_last_cuda_error;

constexpr int kDefaultSms = 152;
constexpr int kDefaultSmemOptin = 232448;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

rgg_status cuda_failure(cudaError_t err, const char* what) {
    g_last_cuda_error = std::string(what) + ": " + cudaGetErrorName(err) + " (" + cudaGetErrorString(err) + ")";
    return RGG_ERR_CUDA;
}

// Makes `device` current for the scope of a call and restores the caller's.
class DeviceScope {
public:
    explicit DeviceScope(int device) {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != device) err_ = cudaSetDevice(device);
    }
    ~DeviceScope() {
        int cur = -1;
        if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
    }
    cudaError_t error() const { return err_; }

private:
    int prev_ = -1;
    cudaError_t err_ = cudaSuccess;
};

using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
    int bm, bn, stages, grid;
    int smem_bytes;
    int64_t max_tiles;
    int tail64;       // 1: tail tiles of <= 64 rows run as 64-row MMAs (128-row tiles only)
    int walk_order;   // 0 list order, 1 front/back interleave, 2 strided scatter, 3 size-sorted, 4 N-major
    // the mixed launch: `grid` / `stages` / `smem_bytes` are the pair kernel's
    // (grid 0: no pair kernel), these the 1-CTA kernel's (grid 0: none)
    int mixed = 0;
    int single_grid = 0, single_stages = 0, single_smem = 0;
    int pair_min_rows = 0;
    // fixed walks only: both kernels launched over all `split_sms` SMs, each
    // CTA computing the split from the device offsets (CTAs past their
    // kernel's share leave at once)
    int device_split = 0, split_sms = 0;
};



// Upper bound on the flat tile count: sum_e ceil(m_e/BM) <= floor(M_tot/BM) + E.
int64_t tile_bound(int E, int64_t M_tot, int N, int bm, int bn) {
    return (M_tot / bm + E) * ceil_div(N, bn);
}

rgg_status check_sizes(int E, int64_t M_tot, int K, int N) {
    if (E < 1 || E > rgg::kMaxExperts) return E < 1 ? RGG_ERR_INVALID_ARG : RGG_ERR_UNSUPPORTED;
    if (M_tot < 0 || M_tot >= (int64_t(1) << 31)) return RGG_ERR_INVALID_ARG;
    if (K < 8 || N < 8 || (K % 8) != 0 || (N % 8) != 0) return RGG_ERR_INVALID_ARG;
    return RGG_OK;
}

// Stages that fit beside a shared-memory carve-up whose fixed part is
// `fixed` bytes, for stages of `per_stage` bytes (tiles + two barriers).
int stages_that_fit(int smem_optin, uint32_t fixed, int64_t per_stage) {
    const int64_t room = static_cast<int64_t>(smem_optin) - 1024 - fixed - 64;
    return static_cast<int>(std::min<int64_t>(rgg::kMaxStages, room / per_stage));
}

// The mixed launch (csrc/rgg_sched.cuh): experts of at least pair_min_rows
// rows on CTA pairs in 256 x 256 tiles, the rest on single CTAs in 128 x 256
// tiles, two kernels on disjoint SMs.  The split of the SMs follows the
// estimated work of each class (mixed_pair_sms in rgg_sched.cuh; with it, 88
// of 152 SMs on pairs for the skewed 16k workload, the measured best: 906
// TFLOP/s against 876 for 84, 872 for 80, 882 for 92, 824 for 100).  With
// claims the kernels steal each other's tiles when their own class runs out,
// so an inexact split costs only the less efficient shape on the stolen
// tiles; the fixed walks depend on it.  Without host counts the fixed walks
// take the split from the device offsets (both kernels launched over all the
// SMs; each CTA computes the same split, and those past their kernel's share
// leave at once), claims take the experts as balanced.
rgg_status plan_mixed(int grid_cap, int smem_optin, int E, int64_t M_tot, int N, const rgg_options* opt, Plan* out,
                      int mode) {
    const int want_bm = opt ? opt->bm : 0;
    const int want_bn = opt ? opt->bn : 0;
    const int want_tail = opt ? opt->tail64 : 0;
    const int want_stages = opt ? opt->stages : 0;
    const int want_psms = opt ? opt->mixed_pair_sms : 0;
    const int pmin = (opt && opt->pair_min_rows > 0) ? opt->pair_min_rows : rgg::kPairMinRowsDefault;
    if ((want_bm != 0 && want_bm != 256) || (want_bn != 0 && want_bn != 256) || want_tail == -1)
        return RGG_ERR_INVALID_ARG;
    if (want_psms < -1 || want_psms > grid_cap || (want_psms > 0 && want_psms % 2 != 0)) return RGG_ERR_INVALID_ARG;
    if (tile_bound(E, M_tot, N, 128, rgg::kMixedBN) >= (int64_t(1) << 31)) return RGG_ERR_UNSUPPORTED;
    const bool host_counts = opt && opt->host_counts;
    const bool device_split = (mode == 2 && want_psms == 0 && !host_counts && grid_cap >= 2);
    int pair_sms = 0;
    if (want_psms == -1) {
        pair_sms = 0;
    } else if (want_psms > 0) {
        pair_sms = want_psms;
    } else {
        const rgg::MixedColCosts cc = rgg::mixed_col_costs(N);
        int64_t cost_p = 0, cost_s = 0;
        if (host_counts) {
            for (int e = 0; e < E; ++e) rgg::mixed_add_expert(cc, opt->host_counts[e], pmin, &cost_p, &cost_s);
        } else {
            int64_t cp = 0, cs = 0;
            rgg::mixed_add_expert(cc, M_tot / E, pmin, &cp, &cs);
            cost_p = cp * E;
            cost_s = cs * E;
        }
        pair_sms = rgg::mixed_pair_sms(cost_p, cost_s, grid_cap);
    }
    pair_sms = std::min(pair_sms, grid_cap & ~1);
    int single = grid_cap - pair_sms;
    if (device_split) {
        pair_sms = grid_cap & ~1;
        single = grid_cap;
    }
    if (pair_sms == 0 && single == 0) return RGG_ERR_INVALID_ARG;

    // shared memory: each kernel keeps the offsets, both class prefixes and the tile queue
    const rgg::SmemPlan pp = rgg::smem_plan(128, 128, 0, E, false, true);
    const rgg::SmemPlan ps = rgg::smem_plan(128, rgg::kMixedBN, 0, E, false, true);
    const int fit_p = stages_that_fit(smem_optin, pp.total, (128 + 128) * 128 + 16);
    const int fit_s = stages_that_fit(smem_optin, ps.total, (128 + rgg::kMixedBN) * 128 + 16);
    const int st_p = want_stages ? want_stages : fit_p;
    const int st_s = want_stages ? want_stages : fit_s;
    if (st_p < 2 || st_p > fit_p || st_s < 2 || st_s > fit_s) return RGG_ERR_UNSUPPORTED;
    const int smem_p = std::max<int>(static_cast<int>(rgg::smem_plan(128, 128, st_p, E, false, true).total) + 1024,
                                     smem_optin / 2 + 1024);
    const int smem_s = std::max<int>(
        static_cast<int>(rgg::smem_plan(128, rgg::kMixedBN, st_s, E, false, true).total) + 1024,
        smem_optin / 2 + 1024);
    if (smem_p > smem_optin || smem_s > smem_optin) return RGG_ERR_UNSUPPORTED;
    out->bm = 256;
    out->bn = rgg::kMixedBN;
    out->stages = st_p;
    out->grid = pair_sms;
    out->smem_bytes = smem_p;
    out->max_tiles = tile_bound(E, M_tot, N, 128, rgg::kMixedBN);
    out->tail64 = 1;
    out->walk_order = 0;
    out->mixed = mode;
    out->single_grid = single;
    out->single_stages = st_s;
    out->single_smem = smem_s;
    out->pair_min_rows = pmin;
    out->device_split = device_split ? 1 : 0;
    out->split_sms = grid_cap;
    return RGG_OK;
}

// Restrictions of the kernel family a plan is for.  kPlanNoPair: 1-CTA
// tiles only (64 or 128 rows); kPlanNoBn192: BN is 128 or 256.  The FP8 op
// (1-CTA tiles only: on CTA pairs it measured slower than 128 x 256 tiles on
// every benchmark shape -- uniform 1 191 vs 1 390 TFLOP/s, skew16k 1 069 vs
// 1 291, prefill 2 714 vs 2 775 -- so it has no pair form) and the fused
// token gather take both; the fused gate-up + SiLU op (N then counts the 2N
// weight columns) takes kPlanNoBn192; the plain token-gather GEMM kPlanNoPair.
constexpr int kPlanNoPair = 1;
constexpr int kPlanNoBn192 = 2;
constexpr int kPlanFused = kPlanNoPair | kPlanNoBn192;

rgg_status make_plan(int num_sms, int smem_optin, int E, int64_t M_tot, int K, int N, const rgg_options* opt,
                     Plan* out, int kind = 0) {
    const bool no_pair = (kind & kPlanNoPair) != 0;
    const bool no_192 = (kind & kPlanNoBn192) != 0;
    rgg_status s = check_sizes(E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (num_sms <= 0) num_sms = kDefaultSms;
    if (smem_optin <= 0) smem_optin = kDefaultSmemOptin;
    const int want_bm = opt ? opt->bm : 0;
    const int want_bn = opt ? opt->bn : 0;
    const int want_stages = opt ? opt->stages : 0;
    const int max_ctas = opt ? opt->max_ctas : 0;
    if (want_bm != 0 && want_bm != 64 && want_bm != 128 && want_bm != 256) return RGG_ERR_INVALID_ARG;
    if (want_bn != 0 && want_bn != 128 && want_bn != 192 && want_bn != 256) return RGG_ERR_INVALID_ARG;
    if (want_bm == 256 && want_bn == 192) return RGG_ERR_INVALID_ARG;  // pair tiles split BN in whole panels
    if ((no_pair && want_bm == 256) || (no_192 && want_bn == 192)) return RGG_ERR_INVALID_ARG;
    if (want_stages != 0 && (want_stages < 2 || want_stages > rgg::kMaxStages)) return RGG_ERR_INVALID_ARG;
    if (max_ctas < 0) return RGG_ERR_INVALID_ARG;
    const int want_tail = opt ? opt->tail64 : 0;
    if (want_tail < -1 || want_tail > 1) return RGG_ERR_INVALID_ARG;
    const int want_walk = opt ? opt->walk_order : 0;
    if (want_walk < -1 || want_walk > 4) return RGG_ERR_INVALID_ARG;  // -1: list order, never replaced
    if (want_walk == 3 && E > rgg::kMaxSortedExperts) return RGG_ERR_UNSUPPORTED;
    int grid_cap = max_ctas > 0 ? std::min(max_ctas, num_sms) : num_sms;
    const int want_mixed = opt ? opt->mixed : 0;
    if (want_mixed < -1 || want_mixed > 2 || (opt && opt->pair_min_rows < 0)) return RGG_ERR_INVALID_ARG;
    if (want_mixed >= 1) {
        if ((kind & ~kPlanNoBn192) != 0) return RGG_ERR_UNSUPPORTED;  // bf16 plain or fused gate-up only
        return plan_mixed(grid_cap, smem_optin, E, M_tot, N, opt, out, want_mixed);
    }

    // Per-expert M tiles at each BM: exact with host counts, else the
    // balanced estimate E * ceil(avg / BM).
    auto m_tiles = [&](int bm) -> int64_t {
        if (opt && opt->host_counts) {
            int64_t t = 0;
            for (int e = 0; e < E; ++e) t += ceil_div(std::max<int64_t>(0, opt->host_counts[e]), bm);
            return t;
        }
        const int64_t avg = ceil_div(M_tot, E);
        return static_cast<int64_t>(E) * ceil_div(avg, bm);
    };

    // Tile shape.  Experts that average 64 rows or fewer (counting only the
    // experts that have rows, when the counts are known) take 64-row tiles:
    // the weight-bound regime, where half-size X stages leave more of the
    // ring to weights.  Otherwise every (BM, BN) candidate is costed as the
    // number of waves of persistent work times a per-tile cost of (BN + 64)
    // (MMA and weight bytes grow with BN, plus a fixed per-tile cost); a CTA
    // pair's 256-row tile occupies two SMs and halves each CTA's weight
    // stage, which measured as 0.87 of a 1-CTA tile of the same BN.  Ties go
    // to the wider tile.  Without host counts the experts are assumed
    // balanced, as in the worklog's eta estimate.
    double avg = static_cast<double>(M_tot) / E;
    if (opt && opt->host_counts) {
        int64_t rows = 0, busy = 0;
        for (int e = 0; e < E; ++e)
            if (opt->host_counts[e] > 0) {
                rows += opt->host_counts[e];
                ++busy;
            }
        avg = busy ? static_cast<double>(rows) / busy : 0.0;
    }
    int bm = want_bm;
    int bn = want_bn;
    if (bm == 0 && avg <= 64.0) bm = 64;
    // 64-row tiles without host counts: 256 columns.  The balanced estimate
    // of the tile count can tip the wave model to 192 columns, which streams
    // the weights in more, smaller tiles (measured on the skewed 2k workload
    // planned from the device offsets: 64 x 192 170 TFLOP/s, 64 x 256 184.5,
    // the host-count plan 184.7; decode already takes 256).
    if (bm == 64 && bn == 0 && want_bm == 0 && !(opt && opt->host_counts)) bn = 256;
    {
        double best = 1e300;
        int best_bm = bm, best_bn = bn;
        for (int cbm : {256, 128, 64}) {
            if (bm != 0 && cbm != bm) continue;
            if (no_pair && cbm == 256) continue;
            if (bm == 0 && cbm == 64) continue;  // 64-row tiles only for small groups (above)
            const bool cpair = (cbm == 256);
            const int cunits = cpair ? std::max(1, grid_cap / 2) : grid_cap;
            const int64_t mt = std::max<int64_t>(1, m_tiles(cbm));
            for (int cbn : {256, 192, 128}) {
                if (bn != 0 && cbn != bn) continue;
                if ((cpair || no_192) && cbn == 192) continue;
                const int64_t waves = ceil_div(mt * ceil_div(N, cbn), cunits);
                const double cost = static_cast<double>(waves) * (cbn + 64) * (cpair ? 0.87 : 1.0);
                if (cost < best) {
                    best = cost;
                    best_bm = cbm;
                    best_bn = cbn;
                }
            }
        }
        bm = best_bm;
        bn = best_bn;
    }
    const bool pair = (bm == 256);
    // Walk order: with the counts known and a strong skew (the largest expert
    // holding over four times the mean of the busy experts), the size-sorted
    // interleave runs tiles of big experts beside tiles of small ones.
    // Otherwise, when experts average three M tiles or more, each expert's
    // tiles are walked N-major (4), so the M tiles that read one weight panel
    // run side by side and the panel is read from HBM once (measured on
    // prefill, E = 32, ~1 024 rows per expert: DRAM reads 3.42 -> 2.73 GB per
    // launch, 1 394 -> 1 408-1 442 TFLOP/s on CTA pairs, FP8 2 801 -> 2 952,
    // fused gate-up 1 408 -> 1 436; with two M tiles per expert, FP8 uniform,
    // it lost 3 %: 1 415 -> 1 373).
    int walk = want_walk;
    bool skewed = false;
    const bool keep_list = (want_walk == -1);
    if (keep_list) walk = 0;
    if (walk == 0 && !keep_list && opt && opt->host_counts && E <= rgg::kMaxSortedExperts) {
        int64_t mx = 0;
        for (int e = 0; e < E; ++e) mx = std::max<int64_t>(mx, opt->host_counts[e]);
        skewed = (avg > 0.0 && static_cast<double>(mx) > 4.0 * avg);
        if (skewed) walk = 3;
    }
    if (walk == 0 && !keep_list && !skewed && avg >= 3.0 * bm) walk = 4;
    // Large experts on CTA pairs, walked N-major: the mixed launch instead
    // (its pair kernel; the 1-CTA kernel only if host counts show small
    // experts), whose tiles are claimed in list order from a device counter.
    // The M tiles that share a weight panel then run side by side whatever
    // the drift between SMs: measured on prefill (E = 32, ~1 024 rows per
    // expert, K = 6144), DRAM reads of 2.75-2.92 GB per launch against 2.07 GB
    // (2.28 GB algorithmic in all), 1 444-1 466 -> 1 494-1 507 TFLOP/s; the
    // fused gate-up op 1 474 -> 1 522-1 548.  Where experts fill only one or
    // two M tiles the static walk stays ahead (uniform 256 rows per expert:
    // 1 093-1 108 static, 1 048 claimed).
    const bool mixed_kind = (kind & ~kPlanNoBn192) == 0;  // the plain and fused gate-up bf16 ops
    if (want_mixed == 0 && mixed_kind && pair && bn == 256 && walk == 4 && want_walk == 0 && want_tail != -1 &&
        (want_stages == 0))
        return plan_mixed(grid_cap, smem_optin, E, M_tot, N, opt, out, 1);
    // Without host counts, experts that average one to three 256-row tiles
    // (more than 64 rows, fewer than 768): the mixed launch with fixed walks,
    // whose kernels take the split of the SMs from the device offsets, so a
    // skewed routing still runs its large experts on pairs and its small ones
    // on single CTAs while the counts never reach the host.  The plain op
    // only, as below.
    if (want_mixed == 0 && kind == 0 && !(opt && opt->host_counts) && avg > 64.0 && avg < 768.0 && want_bm == 0 &&
        (want_bn == 0 || want_bn == 256) && want_walk == 0 && want_tail != -1 && want_stages == 0 && grid_cap >= 2)
        return plan_mixed(grid_cap, smem_optin, E, M_tot, N, opt, out, 2);
    // A strong skew (host counts: the largest expert above four times the
    // mean) over experts that fill 128-row tiles: the large experts on CTA
    // pairs beside the small ones on single CTAs, each kernel walking its own
    // class (measured on the skewed 16k workload: 855-868 TFLOP/s for the
    // size-sorted 128 x 256 walk, 906 for the mixed launch with fixed walks,
    // 841 with claims, whose descriptor queue costs a few microseconds).  The
    // plain op only: on the fused gate-up op it runs level with the static
    // 128 x 256 walk (870 against 868 TFLOP/s), not ahead.
    if (want_mixed == 0 && kind == 0 && skewed && bm == 128 && want_bm == 0 && (want_bn == 0 || want_bn == 256) &&
        want_walk == 0 && want_tail != -1 && want_stages == 0) {
        Plan mp;
        if (plan_mixed(grid_cap, smem_optin, E, M_tot, N, opt, &mp, 2) == RGG_OK && mp.grid > 0 && mp.single_grid > 0) {
            *out = mp;
            return RGG_OK;
        }
    }
    const int units = pair ? std::max(1, grid_cap / 2) : grid_cap;  // persistent CTAs or CTA pairs

    const int64_t max_tiles = tile_bound(E, M_tot, N, bm, bn);
    if (max_tiles >= (int64_t(1) << 31)) return RGG_ERR_UNSUPPORTED;

    // Per-CTA tile extents: a pair CTA holds 128 rows of A and half of B.
    const int cta_m = pair ? 128 : bm;
    const int cta_n = pair ? bn / 2 : bn;
    // walk order 3 keeps the size order and its tile prefix in shared memory as well
    const bool extra_prefix = (walk == 3);
    const rgg::SmemPlan probe = rgg::smem_plan(cta_m, cta_n, 0, E, extra_prefix);
    const int64_t per_stage = static_cast<int64_t>(cta_m + cta_n) * 128 + 16;  // tiles + two barriers
    const int64_t room = static_cast<int64_t>(smem_optin) - 1024 - probe.total - 64;
    int fit = static_cast<int>(std::min<int64_t>(rgg::kMaxStages, room / per_stage));
    int stages = want_stages ? want_stages : fit;
    if (stages < 2 || stages > fit) return RGG_ERR_UNSUPPORTED;

    const rgg::SmemPlan sp = rgg::smem_plan(cta_m, cta_n, stages, E, extra_prefix);
    // Ask for more than half of the SM's shared memory so that exactly one CTA
    // (and one 2 x BN-column TMEM allocation) lives on each SM.
    const int smem = std::max<int>(static_cast<int>(sp.total) + 1024, smem_optin / 2 + 1024);
    if (smem > smem_optin) return RGG_ERR_UNSUPPORTED;

    out->bm = bm;
    out->bn = bn;
    out->stages = stages;
    out->grid = pair ? static_cast<int>(2 * std::max<int64_t>(1, std::min<int64_t>(units, max_tiles)))
                     : static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(grid_cap, max_tiles)));
    out->smem_bytes = smem;
    out->max_tiles = max_tiles;
    out->tail64 = ((bm == 128 || bm == 256) && want_tail != -1) ? 1 : 0;
    out->walk_order = walk;
    return RGG_OK;
}

// Gather modes of the gather calls (rgg_options.gather_mode).
constexpr int kGatherFused = 1;    // TMA tile::gather4 inside the GEMM's producer
constexpr int kGatherTwoPass = 2;  // a row-gather kernel into a workspace, then the grouped GEMM

int64_t gather_workspace_bytes(int64_t M_tot, int K) { return M_tot * static_cast<int64_t>(K) * 2; }

constexpr double kFusedGatherMaxRows = 24.0;

// The caller's mode, else: fused when the experts that have rows average at
// most kFusedGatherMaxRows of them (the few gathered rows per tile hide under
// the weight stream), two-pass otherwise.  Each fused row fetch is a separate
// 128-byte copy repeated for every N tile, and on a GB300 such fetches top
// out near 1.8 TB/s per GPU, a third of what whole-tile boxes reach; gathering
// each routed row once and multiplying with whole-tile boxes wins as soon as
// tiles hold more than a couple of dozen rows (measured with 32 experts,
// K = 6144, N = 4096: fused faster at 1 to 16 rows per expert, by 2% at 16;
// two-pass faster at 32 rows, by 3%, and at 64, by 29%).
//
// The two-pass mode needs the caller's workspace: the library never allocates
// inside a call.  *prefers_two_pass says whether the automatic choice would
// take two passes given a workspace; without one it runs the fused mode
// (CTA pairs, which only the two-pass mode reaches, then cannot be asked for).
rgg_status choose_gather_mode(int E, int64_t M_tot, const rgg_options* opt, int* mode, bool* prefers_two_pass) {
    const int want = opt ? opt->gather_mode : 0;
    if (want < 0 || want > 2) return RGG_ERR_INVALID_ARG;
    *prefers_two_pass = (want == kGatherTwoPass);
    if (want != 0) {
        *mode = want;
        return RGG_OK;
    }
    bool two = false;
    if (opt && opt->bm == 256) {  // CTA pairs read whole boxes
        two = true;
    } else {
        double avg = static_cast<double>(M_tot) / E;
        if (opt && opt->host_counts) {
            int64_t rows = 0, busy = 0;
            for (int e = 0; e < E; ++e)
                if (opt->host_counts[e] > 0) {
                    rows += opt->host_counts[e];
                    ++busy;
                }
            avg = busy ? static_cast<double>(rows) / busy : 0.0;
        }
        two = avg > kFusedGatherMaxRows;
    }
    *prefers_two_pass = two;
    const bool have_ws = opt && opt->workspace;
    if (two && !have_ws && opt && opt->bm == 256) return RGG_ERR_INVALID_ARG;
    *mode = (two && have_ws) ? kGatherTwoPass : kGatherFused;
    return RGG_OK;
}

rgg_status encode_maps(const void* X, const void* W, int E, int64_t M_tot, int K, int N, int bm,
                       CUtensorMap* tx, CUtensorMap* tx64, CUtensorMap* tw) {
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) {
        g_last_cuda_error = "cuTensorMapEncodeTiled is not available from the driver";
        return RGG_ERR_CUDA;
    }
    // X: 2-D {K, M_tot}, box {64, rows per CTA}: one 128-byte swizzle row per tile row.
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M_tot)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(bm > 128 ? 128 : bm)};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = "cuTensorMapEncodeTiled(X) failed with CUresult " + std::to_string(static_cast<int>(r));
            return RGG_ERR_CUDA;
        }
        // The same X with a 64-row box, for tiles that hold 64 rows or fewer.
        const cuuint32_t box64[2] = {64, 64};
        r = encode(tx64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box64, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = "cuTensorMapEncodeTiled(X, 64 rows) failed with CUresult " +
                                std::to_string(static_cast<int>(r));
            return RGG_ERR_CUDA;
        }
    }
    // W: 3-D {N, K, E}, box {64, 64, 1}: one 64-column panel of 64 K rows.
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K),
                                    static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(N) * K * 2};
        const cuuint32_t box[3] = {64, 64, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = encode(tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = "cuTensorMapEncodeTiled(W) failed with CUresult " + std::to_string(static_cast<int>(r));
            return RGG_ERR_CUDA;
        }
    }
    return RGG_OK;
}

// FP8 operands: byte tensors with 128-byte boxes (one swizzle row = 128 K
// elements of X, 128 N columns of W).
rgg_status encode_maps_fp8(const void* X8, const void* W8, int E, int64_t M_tot, int K, int N, int bm,
                           CUtensorMap* tx, CUtensorMap* tx64, CUtensorMap* tw) {
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) {
        g_last_cuda_error = "cuTensorMapEncodeTiled is not available from the driver";
        return RGG_ERR_CUDA;
    }
    const cuuint64_t xdims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M_tot)};
    const cuuint64_t xstrides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t estr2[2] = {1, 1};
    const cuuint32_t xbox[2] = {128, static_cast<cuuint32_t>(bm > 128 ? 128 : bm)};  // a pair CTA holds 128 rows
    const cuuint32_t xbox64[2] = {128, 64};
    const cuuint64_t wdims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(E)};
    const cuuint64_t wstrides[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(N) * K};
    const cuuint32_t wbox[3] = {128, 128, 1};
    const cuuint32_t estr3[3] = {1, 1, 1};
    CUresult r = encode(tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(X8), xdims, xstrides, xbox, estr2,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
        r = encode(tx64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(X8), xdims, xstrides, xbox64, estr2,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
        r = encode(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(W8), wdims, wstrides, wbox, estr3,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled(FP8) failed with CUresult " + std::to_string(static_cast<int>(r));
        return RGG_ERR_CUDA;
    }
    return RGG_OK;
}

// The token matrix [T, K] for tile::gather4 loads: box one row high and one
// 128-byte swizzle row wide, so four gathered rows fill one 512-byte block of
// a stage in the same layout a {64, rows} box would give.
rgg_status encode_token_map(const void* Xtok, int64_t T, int K, CUtensorMap* tx) {
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) {
        g_last_cuda_error = "cuTensorMapEncodeTiled is not available from the driver";
        return RGG_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(Xtok), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled(X_tok) failed with CUresult " +
                            std::to_string(static_cast<int>(r));
        return RGG_ERR_CUDA;
    }
    return RGG_OK;
}

// The token-gather GEMM, plain (Y = X_tok[row_index] . W_e) or with the fused
// gate-up + SiLU epilogue (W then holds 2N columns and Y is H [M_tot, N]).
rgg_status gather_call(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index, const void* W,
                       const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N, void* stream,
                       const rgg_options* opt, bool swiglu);

}  // namespace

namespace rgg {

// Host helpers shared with the other C-ABI translation unit (rgg_noalloc.cu).
rgg_status host_cuda_failure(cudaError_t err, const char* what) { return cuda_failure(err, what); }

void host_set_last_error(const char* what) { g_last_cuda_error = what; }

rgg_status host_check_gemm_args(const void* X, const void* W, const int32_t* group_offsets, const void* Y, int E,
                                int64_t M_tot, int K, int N) {
    if (!group_offsets || !W) return RGG_ERR_INVALID_ARG;
    rgg_status s = check_sizes(E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (M_tot > 0 && (!X || !Y)) return RGG_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(group_offsets, 4) || (M_tot > 0 && (!aligned(X, 16) || !aligned(Y, 16))))
        return RGG_ERR_INVALID_ARG;
    return RGG_OK;
}

rgg_status host_grouped_gemm(int num_sms, int smem_optin, int32_t* status, const void* X, const void* W,
                             const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N,
                             cudaStream_t st, const rgg_options* opt) {
    if (M_tot == 0) {
        cudaError_t err = launch_validate_offsets(group_offsets, E, M_tot, status, st);
        return err == cudaSuccess ? RGG_OK : cuda_failure(err, "validate_offsets launch");
    }
    Plan p;
    rgg_status s = make_plan(num_sms, smem_optin, E, M_tot, K, N, opt, &p, 0);
    if (s != RGG_OK) return s;
    CUtensorMap tx, tx64, tw;
    s = encode_maps(X, W, E, M_tot, K, N, p.bm, &tx, &tx64, &tw);
    if (s != RGG_OK) return s;
    GemmArgs a;
    a.offsets = group_offsets;
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.status = status;
    a.M_tot = M_tot;
    a.E = E;
    a.K = K;
    a.N = N;
    a.num_k_blocks = static_cast<int32_t>(ceil_div(K, kBK));
    a.n_tiles_n = static_cast<int32_t>(ceil_div(N, p.bn));
    a.stages = p.stages;
    a.y_vec32 = ((N % 16) == 0 && aligned(Y, 32)) ? 1 : 0;
    a.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    a.debug_flags = opt ? (opt->debug_flags & RGG_DEBUG_PRODUCER_STALL) : 0;
    a.tail64 = p.tail64;
    a.walk_order = p.walk_order;
    if (p.mixed) {
        // the claim counters and the count of finished CTAs sit 64 bytes after the status word; they
        // start at zero and the launch's last CTA sets them back to zero
        a.sched = status + 16;
        a.sched_total = p.grid + p.single_grid;
        a.sched_pairs = p.grid / 2;
        a.sched_singles = p.single_grid;
        a.sched_claims = (p.mixed == 1) ? 1 : 0;
        a.pair_min_rows = p.pair_min_rows;
        a.sched_split = p.device_split;
        a.split_sms = p.split_sms;
        GemmArgs as = a;
        as.stages = p.single_stages;
        cudaError_t err = launch_gemm_mixed(p.grid, p.smem_bytes, a, p.single_grid, p.single_smem, as, st, tx, tx64,
                                            tw);
        if (err != cudaSuccess) {
            // a kernel that did launch still counts its CTAs: zero the counters behind it
            cudaMemsetAsync(a.sched, 0, 3 * sizeof(int32_t), st);
            return cuda_failure(err, "grouped_gemm (mixed) launch");
        }
        return RGG_OK;
    }
    cudaError_t err = (p.bm == 256)   ? launch_gemm_pair(p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a)
                      : (p.bm == 128) ? launch_gemm_bm128(p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a)
                                      : launch_gemm_bm64(p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a);
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "grouped_gemm launch");
}

}  // namespace rgg

extern "C" {

const char* rgg_status_string(rgg_status s) {
    switch (s) {
        case RGG_OK: return "RGG_OK";
        case RGG_ERR_INVALID_ARG: return "RGG_ERR_INVALID_ARG: invalid argument";
        case RGG_ERR_UNSUPPORTED: return "RGG_ERR_UNSUPPORTED: request not supported by this build or device";
        case RGG_ERR_CUDA: return "RGG_ERR_CUDA: a CUDA call failed";
        case RGG_ERR_BAD_OFFSETS: return "RGG_ERR_BAD_OFFSETS: group offsets are not valid; nothing was written";
        case RGG_ERR_DEVICE_TIMEOUT: return "RGG_ERR_DEVICE_TIMEOUT: a device pipeline wait exceeded its limit";
        case RGG_ERR_CAPACITY: return "RGG_ERR_CAPACITY: more tiles than the output capacity";
        case RGG_ERR_BAD_ROW_INDEX: return "RGG_ERR_BAD_ROW_INDEX: a token index is outside [0, T)";
        case RGG_ERR_DEVICE_BOUNDS:
            return "RGG_ERR_DEVICE_BOUNDS: a device access failed its bounds check (debug build) and was skipped";
    }
    return "unknown rgg_status";
}

const char* rgg_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

rgg_status rgg_create(rgg_handle** out, int device) {
    if (!out) return RGG_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    cudaError_t err = cudaGetDeviceCount(&count);
    if (err != cudaSuccess) return cuda_failure(err, "cudaGetDeviceCount");
    if (device < 0 || device >= count) return RGG_ERR_INVALID_ARG;
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) != cudaSuccess)
        return cuda_failure(err, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
        g_last_cuda_error = "librgg is built for sm_103a; device " + std::to_string(device) + " is sm_" +
                            std::to_string(major) + std::to_string(minor);
        return RGG_ERR_UNSUPPORTED;
    }
    DeviceScope scope(device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    int32_t* status = nullptr;
    if ((err = cudaMalloc(&status, 256)) != cudaSuccess) return cuda_failure(err, "cudaMalloc(status)");
    if ((err = cudaMemset(status, 0, 256)) != cudaSuccess) {
        cudaFree(status);
        return cuda_failure(err, "cudaMemset(status)");
    }
    rgg_handle* h = new rgg_handle;
    h->device = device;
    h->num_sms = sms;
    h->smem_optin = smem;
    h->d_status = status;
    *out = h;
    return RGG_OK;
}

void rgg_destroy(rgg_handle* h) {
    if (!h) return;
    {
        DeviceScope scope(h->device);
        cudaFree(h->d_status);
    }
    delete h;
}

rgg_status rgg_plan(int num_sms, int smem_optin, int E, int64_t M_tot, int K, int N, const rgg_options* opt,
                    rgg_plan_info* out) {
    if (!out) return RGG_ERR_INVALID_ARG;
    Plan p;
    const int op = opt ? opt->op : 0;
    if (op < 0 || op > 4) return RGG_ERR_INVALID_ARG;
    const bool swiglu = (op == 1 || op == 4);
    if (swiglu && (N < 8 || N % 8 != 0 || N > (1 << 30))) return RGG_ERR_INVALID_ARG;
    if (op == 2 && (K % 16 != 0 || N % 16 != 0)) return RGG_ERR_INVALID_ARG;
    const bool gather = (op == 3 || op == 4);
    int mode = 0;
    bool prefers_two_pass = false;
    if (gather) {
        rgg_status sm = choose_gather_mode(E, M_tot, opt, &mode, &prefers_two_pass);
        if (sm != RGG_OK) return sm;
    }
    // the two-pass gather runs the plain (or fused gate-up) kernel on the gathered rows; the fused
    // gate-up op takes CTA pairs but not BN = 192; FP8 and the fused gather take 1-CTA tiles only
    const bool fused_gather = gather && mode == kGatherFused;
    const int kind = (op == 2)                   ? kPlanFused
                     : (op == 4 && fused_gather) ? kPlanFused
                     : (op == 3 && fused_gather) ? kPlanNoPair
                     : swiglu                    ? kPlanNoBn192
                                                 : 0;
    rgg_status s = make_plan(num_sms, smem_optin, E, M_tot, K, swiglu ? 2 * N : N, opt, &p, kind);
    if (s != RGG_OK) return s;
    out->bm = p.bm;
    out->bn = p.bn;
    out->bk = (op == 2) ? 128 : rgg::kBK;
    out->stages = p.stages;
    out->grid = p.grid;
    // FP8 and the fused gate-up op run eight epilogue warps (on CTA pairs: per CTA)
    out->threads = (op == 2 || swiglu) ? rgg::cta_threads<rgg::kEpiSwiGLU, false>() : rgg::kThreads;  // 320 or 192
    out->smem_bytes = p.smem_bytes;
    out->tmem_cols = (p.bm == 256 || 2 * p.bn > 256) ? 512 : 256;
    out->max_tiles = p.max_tiles;
    out->tail64 = p.tail64;
    out->walk_order = p.walk_order;
    if (swiglu && p.bm == 256 && p.bn != 256) out->tail64 = 0;  // 128-column gate-up pairs keep 256-row tails
    out->gather_mode = mode;
    out->workspace_bytes = prefers_two_pass ? gather_workspace_bytes(M_tot, K) : 0;
    out->mixed = p.mixed;
    out->single_grid = p.single_grid;
    out->single_stages = p.single_stages;
    out->single_smem_bytes = p.single_smem;
    out->pair_min_rows = p.pair_min_rows;
    out->device_split = p.device_split;
    if (p.mixed) out->tmem_cols = 512;
    return RGG_OK;
}

rgg_status rgg_grouped_gemm(rgg_handle* h, const void* X, const void* W, const int32_t* group_offsets, void* Y,
                            int E, int64_t M_tot, int K, int N, void* stream, const rgg_options* opt) {
    if (!h) return RGG_ERR_INVALID_ARG;
    rgg_status s = rgg::host_check_gemm_args(X, W, group_offsets, Y, E, M_tot, K, N);
    if (s != RGG_OK) return s;
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    return rgg::host_grouped_gemm(h->num_sms, h->smem_optin, h->d_status, X, W, group_offsets, Y, E, M_tot, K, N,
                                  static_cast<cudaStream_t>(stream), opt);
}

rgg_status rgg_grouped_gemm_swiglu(rgg_handle* h, const void* X, const void* W13, const int32_t* group_offsets,
                                   void* H, int E, int64_t M_tot, int K, int N, void* stream,
                                   const rgg_options* opt) {
    if (!h || !group_offsets || !W13) return RGG_ERR_INVALID_ARG;
    rgg_status s = check_sizes(E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (N > (1 << 30)) return RGG_ERR_INVALID_ARG;
    if (M_tot > 0 && (!X || !H)) return RGG_ERR_INVALID_ARG;
    if (!aligned(W13, 16) || !aligned(group_offsets, 4) || (M_tot > 0 && (!aligned(X, 16) || !aligned(H, 16))))
        return RGG_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    if (M_tot == 0) {
        cudaError_t err = rgg::launch_validate_offsets(group_offsets, E, M_tot, h->d_status, st);
        return err == cudaSuccess ? RGG_OK : cuda_failure(err, "validate_offsets launch");
    }
    Plan p;
    s = make_plan(h->num_sms, h->smem_optin, E, M_tot, K, 2 * N, opt, &p, kPlanNoBn192);
    if (s != RGG_OK) return s;
    CUtensorMap tx, tx64, tw;
    s = encode_maps(X, W13, E, M_tot, K, 2 * N, p.bm, &tx, &tx64, &tw);
    if (s != RGG_OK) return s;
    rgg::GemmArgs a;
    a.offsets = group_offsets;
    a.Y = static_cast<__nv_bfloat16*>(H);
    a.status = h->d_status;
    a.M_tot = M_tot;
    a.E = E;
    a.K = K;
    a.N = N;  // output columns; the gate / up split of W13 is at column N
    a.num_k_blocks = static_cast<int32_t>(ceil_div(K, rgg::kBK));
    a.n_tiles_n = static_cast<int32_t>(ceil_div(N, p.bn / 2));
    a.stages = p.stages;
    a.y_vec32 = ((N % 16) == 0 && aligned(H, 32)) ? 1 : 0;
    a.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    a.debug_flags = opt ? (opt->debug_flags & RGG_DEBUG_PRODUCER_STALL) : 0;
    a.tail64 = p.tail64;
    a.walk_order = p.walk_order;
    if (p.mixed) {
        // as for rgg_grouped_gemm's mixed launch
        a.sched = h->d_status + 16;
        a.sched_total = p.grid + p.single_grid;
        a.sched_pairs = p.grid / 2;
        a.sched_singles = p.single_grid;
        a.sched_claims = (p.mixed == 1) ? 1 : 0;
        a.pair_min_rows = p.pair_min_rows;
        a.sched_split = p.device_split;
        a.split_sms = p.split_sms;
        rgg::GemmArgs as = a;
        as.stages = p.single_stages;
        cudaError_t err = rgg::launch_gemm_mixed_swiglu(p.grid, p.smem_bytes, a, p.single_grid, p.single_smem, as, st,
                                                        tx, tx64, tw);
        if (err != cudaSuccess) {
            cudaMemsetAsync(a.sched, 0, 3 * sizeof(int32_t), st);
            return cuda_failure(err, "grouped_gemm_swiglu (mixed) launch");
        }
        return RGG_OK;
    }
    if (p.bm == 256 && p.bn != 256) a.tail64 = 0;  // 128-column pairs: a 64-column panel cannot hold gate and up
    cudaError_t err = (p.bm == 256) ? rgg::launch_gemm_pair_swiglu(p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a)
                                    : rgg::launch_gemm_swiglu(p.bm, p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a);
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "grouped_gemm_swiglu launch");
}

rgg_status rgg_grouped_gemm_fp8(rgg_handle* h, const void* X8, const void* W8, const float* sx, const float* sw,
                                const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N,
                                void* stream, const rgg_options* opt) {
    if (!h || !group_offsets || !W8 || !sw) return RGG_ERR_INVALID_ARG;
    rgg_status s = check_sizes(E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (K < 16 || N < 16 || K % 16 != 0 || N % 16 != 0) return RGG_ERR_INVALID_ARG;
    if (M_tot > 0 && (!X8 || !Y || !sx)) return RGG_ERR_INVALID_ARG;
    if (!aligned(W8, 16) || !aligned(sw, 16) || !aligned(group_offsets, 4) ||
        (M_tot > 0 && (!aligned(X8, 16) || !aligned(Y, 16) || !aligned(sx, 4))))
        return RGG_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    if (M_tot == 0) {
        cudaError_t err = rgg::launch_validate_offsets(group_offsets, E, M_tot, h->d_status, st);
        return err == cudaSuccess ? RGG_OK : cuda_failure(err, "validate_offsets launch");
    }
    Plan p;
    s = make_plan(h->num_sms, h->smem_optin, E, M_tot, K, N, opt, &p, kPlanFused);
    if (s != RGG_OK) return s;
    CUtensorMap tx, tx64, tw;
    s = encode_maps_fp8(X8, W8, E, M_tot, K, N, p.bm, &tx, &tx64, &tw);
    if (s != RGG_OK) return s;
    rgg::GemmArgs a;
    a.offsets = group_offsets;
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.status = h->d_status;
    a.M_tot = M_tot;
    a.E = E;
    a.K = K;
    a.N = N;
    a.num_k_blocks = static_cast<int32_t>(ceil_div(K, 128));
    a.n_tiles_n = static_cast<int32_t>(ceil_div(N, p.bn));
    a.stages = p.stages;
    a.y_vec32 = ((N % 16) == 0 && aligned(Y, 32)) ? 1 : 0;
    a.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    a.debug_flags = opt ? (opt->debug_flags & RGG_DEBUG_PRODUCER_STALL) : 0;
    a.tail64 = p.tail64;
    a.walk_order = p.walk_order;
    a.sx = sx;
    a.sw = sw;
    cudaError_t err = rgg::launch_gemm_fp8(p.bm, p.bn, p.grid, p.smem_bytes, st, tx, tx64, tw, a);
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "grouped_gemm_fp8 launch");
}

rgg_status rgg_grouped_gemm_gather(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index,
                                   const void* W, const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K,
                                   int N, void* stream, const rgg_options* opt) {
    return gather_call(h, X_tok, T, row_index, W, group_offsets, Y, E, M_tot, K, N, stream, opt, false);
}

rgg_status rgg_grouped_gemm_swiglu_gather(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index,
                                          const void* W13, const int32_t* group_offsets, void* H, int E,
                                          int64_t M_tot, int K, int N, void* stream, const rgg_options* opt) {
    return gather_call(h, X_tok, T, row_index, W13, group_offsets, H, E, M_tot, K, N, stream, opt, true);
}

rgg_status rgg_export_tiles(rgg_handle* h, const int32_t* group_offsets, int E, int64_t M_tot, int N, int bm,
                            int bn, int32_t* desc_out, int64_t cap, int32_t* n_tiles_out, void* stream) {
    if (!h || !group_offsets || !n_tiles_out || cap < 0 || (cap > 0 && !desc_out)) return RGG_ERR_INVALID_ARG;
    if (E < 1 || E > rgg::kMaxExperts || M_tot < 0 || M_tot >= (int64_t(1) << 31) || N < 1)
        return RGG_ERR_INVALID_ARG;
    if ((bm != 64 && bm != 128 && bm != 256) || (bn != 128 && bn != 192 && bn != 256)) return RGG_ERR_INVALID_ARG;
    if (tile_bound(E, M_tot, N, bm, bn) >= (int64_t(1) << 31)) return RGG_ERR_UNSUPPORTED;
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    cudaError_t err = rgg::launch_export_tiles(group_offsets, E, M_tot, N, bm, bn, 0, desc_out, cap, n_tiles_out,
                                               h->d_status, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "export_tiles launch");
}

rgg_status rgg_export_walk(rgg_handle* h, const int32_t* group_offsets, int E, int64_t M_tot, int N, int bm,
                           int bn, int walk_order, int32_t* desc_out, int64_t cap, int32_t* n_tiles_out,
                           void* stream) {
    if (!h || !group_offsets || !n_tiles_out || cap < 0 || (cap > 0 && !desc_out)) return RGG_ERR_INVALID_ARG;
    if (E < 1 || E > rgg::kMaxExperts || M_tot < 0 || M_tot >= (int64_t(1) << 31) || N < 1)
        return RGG_ERR_INVALID_ARG;
    if ((bm != 64 && bm != 128 && bm != 256) || (bn != 128 && bn != 192 && bn != 256)) return RGG_ERR_INVALID_ARG;
    if (walk_order < 0 || walk_order > 4) return RGG_ERR_INVALID_ARG;
    if (walk_order == 3 && E > rgg::kMaxSortedExperts) return RGG_ERR_UNSUPPORTED;
    if (tile_bound(E, M_tot, N, bm, bn) >= (int64_t(1) << 31)) return RGG_ERR_UNSUPPORTED;
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    cudaError_t err = rgg::launch_export_tiles(group_offsets, E, M_tot, N, bm, bn, walk_order, desc_out, cap,
                                               n_tiles_out, h->d_status, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "export_walk launch");
}

rgg_status rgg_query_status(rgg_handle* h, void* stream) {
    if (!h) return RGG_ERR_INVALID_ARG;
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t value = 0;
    cudaError_t err = cudaMemcpyAsync(&value, h->d_status, sizeof(value), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaMemsetAsync(h->d_status, 0, sizeof(int32_t), st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return cuda_failure(err, "rgg_query_status");
    return static_cast<rgg_status>(value);
}

}  // extern "C"

namespace {

rgg_status gather_call(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index, const void* W,
                       const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N, void* stream,
                       const rgg_options* opt, bool swiglu) {
    if (!h || !group_offsets || !W) return RGG_ERR_INVALID_ARG;
    rgg_status s = check_sizes(E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (swiglu && N > (1 << 30)) return RGG_ERR_INVALID_ARG;
    if (T < 0 || T >= (int64_t(1) << 31)) return RGG_ERR_INVALID_ARG;
    if (M_tot > 0 && (!X_tok || !row_index || !Y || T < 1)) return RGG_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(group_offsets, 4) ||
        (M_tot > 0 && (!aligned(X_tok, 16) || !aligned(Y, 16) || !aligned(row_index, 4))))
        return RGG_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceScope scope(h->device);
    if (scope.error() != cudaSuccess) return cuda_failure(scope.error(), "cudaSetDevice");
    if (M_tot == 0) {
        cudaError_t err = rgg::launch_validate_offsets(group_offsets, E, M_tot, h->d_status, st);
        return err == cudaSuccess ? RGG_OK : cuda_failure(err, "validate_offsets launch");
    }
    const int NW = swiglu ? 2 * N : N;  // weight columns
    int mode = 0;
    bool prefers_two_pass = false;
    s = choose_gather_mode(E, M_tot, opt, &mode, &prefers_two_pass);
    if (s != RGG_OK) return s;
    if (mode == kGatherTwoPass) {
        // Pass 1 writes the routed rows, in routed order, into the caller's
        // workspace; pass 2 is the grouped product of those rows.
        const int64_t need = gather_workspace_bytes(M_tot, K);
        void* ws = opt ? opt->workspace : nullptr;
        if (!ws || opt->workspace_bytes < need || !aligned(ws, 16)) return RGG_ERR_INVALID_ARG;
        cudaError_t err = rgg::launch_gather_rows(X_tok, row_index, group_offsets, E, M_tot, T, K, ws, h->num_sms,
                                                  h->d_status, st);
        if (err != cudaSuccess) return cuda_failure(err, "gather_rows launch");
        return swiglu ? rgg_grouped_gemm_swiglu(h, ws, W, group_offsets, Y, E, M_tot, K, N, stream, opt)
                      : rgg_grouped_gemm(h, ws, W, group_offsets, Y, E, M_tot, K, N, stream, opt);
    }
    Plan p;
    s = make_plan(h->num_sms, h->smem_optin, E, M_tot, K, NW, opt, &p, swiglu ? kPlanFused : kPlanNoPair);
    if (s != RGG_OK) return s;
    CUtensorMap tx, tx64, tw;
    s = encode_maps(X_tok, W, E, T, K, NW, p.bm, &tx, &tx64, &tw);  // W map (the X maps are replaced below)
    if (s != RGG_OK) return s;
    s = encode_token_map(X_tok, T, K, &tx);
    if (s != RGG_OK) return s;
    rgg::GemmArgs a;
    a.offsets = group_offsets;
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.status = h->d_status;
    a.M_tot = M_tot;
    a.E = E;
    a.K = K;
    a.N = N;
    a.num_k_blocks = static_cast<int32_t>(ceil_div(K, rgg::kBK));
    a.n_tiles_n = static_cast<int32_t>(ceil_div(N, swiglu ? p.bn / 2 : p.bn));
    a.stages = p.stages;
    a.y_vec32 = ((N % 16) == 0 && aligned(Y, 32)) ? 1 : 0;
    a.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    a.debug_flags = opt ? (opt->debug_flags & RGG_DEBUG_PRODUCER_STALL) : 0;
    a.tail64 = p.tail64;
    a.walk_order = p.walk_order;
    a.row_index = row_index;
    a.t_rows = static_cast<int32_t>(T);
    cudaError_t err = rgg::launch_gemm_gather(swiglu, p.bm, p.bn, p.grid, p.smem_bytes, st, tx, tw, a);
    return err == cudaSuccess ? RGG_OK : cuda_failure(err, "grouped_gemm_gather launch");
}

}  // namespace
