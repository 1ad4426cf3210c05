// rgg_gemm_mc.cuh -- the 1-CTA grouped GEMM on clusters of two CTAs that
// share one operand of each pair of tiles through TMA multicast.
//
// Sources (by page title and section): the tile list, ring, MMA and epilogue
// are those of the 1-CTA kernel (rgg_gemm.cuh); "Grouped GEMM for Imbalanced
// Experts on Blackwell: A WIP Worklog", section 5 (TMA loads into a
// multistage mbarrier ring) and section 7 (one thread per CTA issues
// tcgen05.mma from shared-memory descriptors into TMEM).
//
// Why: on the skewed routings the 1-CTA kernel's time is set by how many bytes
// its SMs pull out of L2 (every tile reads its X rows and its weight panel
// from L2).  Here the two CTAs of a cluster walk two-tile units
// (rgg_tiles.cuh): consecutive M tiles of one expert at the same N tile share
// the weight panel, and neighbouring N tiles of one M tile share the X rows.
// Each CTA loads half of the shared operand with a multicast copy that lands
// in both CTAs' shared memory, so L2 serves that operand once per unit instead
// of twice.  The MMAs stay cta_group::1 (each CTA computes its own 128 x BN
// tile into its own TMEM), so units of different shapes mix freely.
//
// Ring protocol: both CTAs walk the same units, stage for stage.  A stage
// slot of a CTA can be overwritten by either CTA's multicast, so its empty
// barrier takes two arrivals: each CTA's MMA thread commits to the slot's
// empty barrier in both CTAs (tcgen05.commit multicast).  Each CTA arms its
// own full barrier with every byte that lands in its slot (its own copies and
// the other CTA's multicast); the transaction count may run ahead of the
// arming, which the mbarrier allows.
//
// Roles per CTA as in the 1-CTA kernel: warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer, then the epilogue warps.  Every wait is bounded; a timeout
// raises both CTAs' abort flags, copies and MMAs already issued are waited for
// (bounded), and the CTAs meet at a cluster barrier before TMEM is freed.
#pragma once

#include "rgg_gemm.cuh"

namespace rgg {

template <int BN, int kEpi = kEpiPlain, bool kFp8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_threads<kEpi, kFp8>(), 1)
    grouped_gemm_mc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_x64,
                           const __grid_constant__ CUtensorMap tmap_w, const GemmArgs args) {
    constexpr int BM = 128;
    using Cfg = TileConfig<BM, BN, kFp8>;
    static_assert(kEpi == kEpiPlain || (BN % 128) == 0, "fused gate-up tiles hold whole gate and up panels");
    static_assert(!(kFp8 && kEpi == kEpiSwiGLU), "the fused gate-up epilogue is bf16 only");
    constexpr int kOutN = (kEpi == kEpiSwiGLU) ? BN / 2 : BN;
    constexpr int kPanels = BN / Cfg::kPanelN;
    static_assert(kPanels % 2 == 0, "a shared weight stage splits into whole panels, half per CTA");
    constexpr uint32_t kHalfRowsBytes = 64u * 128u;  // 64 rows of an A stage
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
    const int rank = static_cast<int>(cluster_ctarank());
    const int32_t cl = static_cast<int32_t>(cluster_id_x());
    const int32_t ncl = static_cast<int32_t>(cluster_count_x());

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const SmemPlan sp = smem_plan(BM, BN, S, E, true);
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
    int32_t* s_upre = reinterpret_cast<int32_t*>(gbase + sp.pre_off);
    int32_t* s_lpre = reinterpret_cast<int32_t*>(gbase + sp.ord_off);

    // S1, identical in both CTAs, so every early exit below is cluster-uniform.
    if (!load_and_check_offsets(args.offsets, s_off, E, args.M_tot)) {
        if (threadIdx.x == 0 && rank == 0) atomicCAS(args.status, 0, kStatusBadOffsets);
        return;
    }
    if (warp == 0) build_unit_prefix_warp(s_off, s_upre, s_lpre, E, BM, args.n_tiles_n);
    __syncthreads();
    const int32_t U = unit_count(s_upre, s_lpre, E);
    if (cl >= U) return;

    if (threadIdx.x == 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 2);  // one commit from each CTA's MMA thread
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), epilogue_warps<kEpi, kFp8>());
        }
        mbar_init(drain_bar, 1);
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
    cluster_sync_all();  // both CTAs' barriers initialised before any multicast or remote arrival
    tc_fence_after_sync();

    const uint32_t tmem_base = misc[0];
    volatile uint32_t* abort_flag = &misc[1];
    const uint32_t peer_flag = map_to_rank(smem_addr(&misc[1]), static_cast<uint32_t>(rank ^ 1));
    const int KB = args.num_k_blocks;
    const int nN = args.n_tiles_n;
    const int WO = args.walk_order;  // 0, 1 or 2 (the host maps the size-sorted order to 1)
    const int32_t WS = walk_stride_for(U);
    auto unit_at = [&](int32_t p) -> UnitTile {
        return decode_unit(s_off, s_upre, s_lpre, E, BM, kOutN, nN, walk_tile(p, U, WO, WS), rank);
    };

    if (warp == 0) {
        // ---------------------------------------------------- S4: TMA producer
        if (lane == 0 && (args.debug_flags & kDebugProducerStall) == 0) {
            int st = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int32_t p = cl; ok && p < U; p += ncl) {
                const UnitTile ut = unit_at(p);
                const TileCoord& c = ut.c;
                const bool half = runs_as_64_rows<BM>(args, c);
                const CUtensorMap* xmap = half ? &tmap_x64 : &tmap_x;
                const uint32_t tx_bytes = half ? Cfg::kStageTx64 : Cfg::kStageTx;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!pair_wait_or_abort(empty_bar(st), ph ^ 1u, abort_flag, peer_flag, args.status,
                                            args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(st), tx_bytes);
                    const int32_t kx = kb * Cfg::kKStage;
                    const uint32_t a_st = a0 + st * sp.a_stage;
                    const uint32_t b_st = b0 + st * sp.b_stage;
                    if (ut.share == kShareA) {
                        // the same rows in both CTAs: a 64-row box from CTA 0, or 64 rows from each
                        if (half) {
                            if (rank == 0) tma_load_2d_mc(a_st, &tmap_x64, full_bar(st), kx, c.row0, 0x3);
                        } else {
                            tma_load_2d_mc(a_st + kHalfRowsBytes * rank, &tmap_x64, full_bar(st), kx,
                                           c.row0 + 64 * rank, 0x3);
                        }
                    } else {
                        tma_load_2d(a_st, xmap, full_bar(st), kx, c.row0);
                    }
#pragma unroll
                    for (int q = 0; q < kPanels; ++q) {
                        const uint32_t dst = b_st + q * Cfg::kPanelB;
                        if (ut.share == kShareB) {
                            // the same panels in both CTAs: each loads its half for both
                            if ((q < kPanels / 2) == (rank == 0))
                                tma_load_3d_mc(dst, &tmap_w, full_bar(st), w_col(c.col0, q), kx, c.expert, 0x3);
                        } else {
                            tma_load_3d(dst, &tmap_w, full_bar(st), w_col(c.col0, q), kx, c.expert);
                        }
                    }
                    ++issued;
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the bytes headed for the armed stages land (this CTA's and
                // the other's multicast) before the CTA can exit; the whole
                // drain shares one time limit.
                const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
                const uint64_t t_end = global_timer_ns() + kDrainLimitNs;
                for (uint32_t i = issued - n; i < issued; ++i) {
                    const uint64_t now = global_timer_ns();
                    if (now >= t_end) break;
                    wait_bounded(full_bar(static_cast<int>(i % S)), (i / S) & 1u, t_end - now);
                }
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
            for (int32_t p = cl; ok && p < U; p += ncl) {
                const TileCoord c = unit_at(p).c;
                const uint32_t idesc = runs_as_64_rows<BM>(args, c) ? Cfg::kIdesc64 : Cfg::kIdesc;
                if (!pair_wait_or_abort(acce_bar(acc), acc_ph ^ 1u, abort_flag, peer_flag, args.status,
                                        args.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!pair_wait_or_abort(full_bar(st), ph, abort_flag, peer_flag, args.status, args.timeout_ns)) {
                        ok = false;
                        break;
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
                    mma_commit_mc(empty_bar(st), 0x3);  // the slot is free in both CTAs once both have read it
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_ph ^= 1u;
                }
            }
            if (!ok) {
                mma_commit(drain_bar);
                wait_bounded(drain_bar, 0u, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- S6: epilogue
        const int q = warp & 3;
        constexpr int kParts = epilogue_warps<kEpi, kFp8>() / 4;
        constexpr int kPartCols = kOutN / kParts;
        static_assert(kPartCols % 32 == 0, "each epilogue warp handles whole 32-column chunks");
        const int cc0 = ((warp - 2) >> 2) * kPartCols;
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int32_t p = cl; p < U; p += ncl) {
            const UnitTile ut = unit_at(p);
            const bool half = runs_as_64_rows<BM>(args, ut.c);
            const int r_local = half ? (q * 16 + (lane & 15)) : (q * 32 + lane);
            bool ok = pair_wait_or_abort(accf_bar(acc), acc_ph, abort_flag, peer_flag, args.status, args.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            epilogue_store_tile<BN, kEpi, kFp8>(args, ut.c, half, r_local, t_row, lane, cc0, ut.store);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1u;
            }
        }
    }

    tc_fence_before_sync();
    cluster_sync_all();  // neither CTA leaves while the other's multicasts or arrivals may reach it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace rgg
