// rgg_gemm_2cta.cuh -- the CTA-pair (tcgen05 cta_group::2) variant for large
// expert groups: 256-row tiles computed by two CTAs on neighbouring SMs.
//
// "Pearl's grouped GEMM kernel for MoE models, explained", "Four changes,
// three of them measured", describes a baseline library that offers its
// smaller tiles only in a two-block mode; for large groups the pair mode is
// the natural shape on Blackwell: one tcgen05.mma of M = 256 reads the A rows
// of both CTAs (128 each) and the B columns of both CTAs (BN/2 each) and
// writes each CTA's 128 accumulator rows into that CTA's TMEM.  Each CTA
// therefore loads only half of the weight tile per stage, which halves the
// shared-memory fill per FLOP compared with one CTA holding the whole
// 128 x BN tile.  Every CTA loads its own boxes into its own shared memory.
//
// Roles (both CTAs run the same code, rank = %cluster_ctarank):
//   warp 0 lane 0 : producer.  Waits its own empty[s]; the leader (rank 0)
//                   arms its full[s] for both CTAs' bytes; both CTAs' TMA
//                   loads complete on the leader's full[s].
//   warp 1        : allocates the pair's TMEM in both CTAs; lane 0 of the
//                   leader issues every MMA and commits to the empty /
//                   acc_full barriers of both CTAs with one commit.
//   warps 2-5     : epilogue of the CTA's own 128 rows (warps 2-9, two per
//   (or 2-9)        TMEM lane quadrant, for the fused gate-up epilogue);
//                   they arrive on the leader's acc_empty (one arrival per
//                   epilogue warp of both CTAs).
// All waits are bounded; an abort raised in either CTA is mirrored into the
// other CTA's flag so the pair leaves its loops together.
#pragma once

#include "rgg_gemm.cuh"

namespace rgg {

// bf16 stages: K = 64 (one 128-byte swizzle row) with 64-column weight panels.
template <int BN>
struct PairConfig {
    static_assert(BN == 128 || BN == 256, "pair tiles split BN into two whole 64-column panel sets");
    static constexpr int kHalfN = BN / 2;           // B columns held by each CTA
    static constexpr int kKStage = kBK;              // K elements per stage
    static constexpr int kPanelN = 64;               // W columns per panel
    static constexpr int kPanels = kHalfN / kPanelN;
    static constexpr uint32_t kPanelB = static_cast<uint32_t>(kKStage) * 128u;  // bytes per W panel
    static constexpr uint32_t kBStep = 2048u;       // B start advance per MMA (16 K rows)
    static constexpr uint32_t kTmemCols = 512;      // two BN-column fp32 buffers (BN <= 256)
};

// Columns a pair tile multiplies: BN, or for a plain tile whose columns run
// past N (an expert's last N tile) the columns below N rounded up to 128, so
// that each CTA still holds whole 64-column panels (N/2 of them per CTA).
// The copies and MMAs of the columns past that are not issued.
template <int BN, int kEpi>
__device__ __forceinline__ int pair_tile_cols(int32_t col0, int32_t N) {
    if (kEpi != kEpiPlain) return BN;
    const int32_t need = (N - col0 + 127) / 128 * 128;
    return need < BN ? static_cast<int>(need) : BN;
}

// A pair tile whose rows are the last <= 128 of its expert runs as an M = 128
// pair MMA (args.tail64): each CTA loads and computes 64 rows, which halves
// the padded MMA work of small experts while the tile list stays the same.
__device__ __forceinline__ bool pair_runs_as_128_rows(const GemmArgs& args, const TileCoord& c) {
    return args.tail64 != 0 && c.rows <= 128;
}

// kEpi = kEpiSwiGLU: the fused gate-up projection on a pair.  A tile covers
// BN/2 output columns; CTA 0 loads the BN/2 gate columns and CTA 1 the
// matching BN/2 up columns as the two halves of B, so the M = 256 MMA leaves
// [gate | up] side by side in each CTA's TMEM for that CTA's 128 rows, and the
// epilogue writes silu(gate) * up.  A tail tile of <= 128 rows (BN = 256)
// runs as an M = 128 pair MMA, whose accumulator puts the first half of B's
// columns in TMEM lanes 0-63 and the second half in lanes 64-127 (see the
// epilogue); so that each lane holds a gate column and its up column, CTA r
// then loads gate columns [64 r, 64 r + 64) and the matching up columns of
// the tile, and lanes 0-63 / 64-127 produce output columns [0, 64) / [64, 128).
// (BN = 128 keeps tails at M = 256: a 64-column panel cannot be split.)
// Epilogue warps per CTA: four for plain bf16 outputs, eight (two per TMEM
// lane quadrant, each on half of the columns) for the fused gate-up epilogue,
// whose exponentials otherwise outlast the main loop (measured: uniform 845 ->
// 1 018 TFLOP/s, prefill 1 417 -> 1 526).
template <int kEpi>
__host__ __device__ constexpr int pair_epilogue_warps() {
    return kEpi == kEpiSwiGLU ? 8 : 4;
}

// kDyn: the pair kernel of the mixed launch (rgg_sched.cuh).  The leader's
// producer claims tiles from the device counters (class P first, then the
// 1-CTA class as M = 128 pair tiles) and writes each descriptor into both
// CTAs' tile queues; the leader's MMA thread, the peer's producer and both
// CTAs' epilogue warps take it from their own CTA's queue and release the slot
// on the leader's q_empty.  A descriptor with expert -1 ends the walk.
template <int BN, int kEpi = kEpiPlain, bool kDyn = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * pair_epilogue_warps<kEpi>(), 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_x64,
                             const __grid_constant__ CUtensorMap tmap_w, const GemmArgs args) {
    using Cfg = PairConfig<BN>;
    static_assert(!kDyn || BN == kMixedBN, "the mixed launch's pairs run 256-column MMAs");
    constexpr int BM = 256;  // rows per pair tile
    constexpr int kOutN = (kEpi == kEpiSwiGLU) ? BN / 2 : BN;  // output columns per tile
    auto half_tile = [&](const TileCoord& c) {
        return (kEpi == kEpiPlain || BN == 256) && pair_runs_as_128_rows(args, c);
    };
    extern __shared__ __align__(1024) uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = args.E;
    const int S = args.stages;
    const uint32_t rank = cluster_ctarank();
    const uint32_t pair = cluster_id_x();
    const uint32_t npairs = cluster_count_x();

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const SmemPlan sp = smem_plan(128, Cfg::kHalfN, S, E, !kDyn && args.walk_order == 3, kDyn);
    const uint32_t a0 = base + sp.a_off;
    const uint32_t b0 = base + sp.b_off;
    const uint32_t bars = base + sp.bar_off;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + sp.misc_off);
    volatile uint32_t* info_ring = misc + 4;  // static walk: the leader's MMA instruction descriptors (kInfoSlots)
    int32_t* s_off = reinterpret_cast<int32_t*>(gbase + sp.off_off);
    int32_t* s_pre = reinterpret_cast<int32_t*>(gbase + sp.pre_off);
    int32_t* s_order = reinterpret_cast<int32_t*>(gbase + sp.ord_off);  // walk order 3; mixed: class S prefix
    int32_t* s_spre = reinterpret_cast<int32_t*>(gbase + sp.spre_off);
    int32_t* q_desc = reinterpret_cast<int32_t*>(gbase + sp.q_off);     // mixed: tile queue
    auto qfull_bar = [&](int i) { return base + sp.qbar_off + 8u * i; };
    auto qempty_bar = [&](int i) { return base + sp.qbar_off + 8u * (kQueueDepth + i); };

    // No global memory access before the kernel ahead on the stream has
    // finished (programmatic stream serialisation, as in the 1-CTA kernel);
    // then the next grid may launch: the mixed launch's 1-CTA kernel starts
    // beside this one as soon as every pair CTA has got here.
    pdl_wait_prerequisites();
    pdl_launch_dependents();

    // S1, identical in both CTAs, so every early exit below is pair-uniform.
    if (!load_and_check_offsets(args.offsets, s_off, E, args.M_tot)) {
        if (threadIdx.x == 0 && rank == 0) atomicCAS(args.status, 0, kStatusBadOffsets);
        if constexpr (kDyn)
            if (threadIdx.x == 0 && args.sched_claims) sched_cta_done(args.sched, args.sched_total);
        return;
    }
    ClassLists L;
    int32_t T;
    // mixed launch, fixed walks: clusters of this kernel and CTAs of the
    // 1-CTA kernel that take part (cluster k walks positions k, k + units, ...)
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
            return;
        }
        pair_units = args.sched_split ? static_cast<int32_t>(misc[2]) / 2 : args.sched_pairs;
        single_units = args.sched_split ? args.split_sms - static_cast<int32_t>(misc[2]) : args.sched_singles;
        // past this kernel's share (both CTAs of the pair alike): leave
        if (args.sched_split && static_cast<int32_t>(pair) >= pair_units) return;
    } else {
        if (warp == 0) build_tile_prefix_warp(s_off, s_pre, E, BM, args.n_tiles_n);
        __syncthreads();
        T = s_pre[E];
        if (args.walk_order == 3) build_size_order(s_off, s_order, s_spre, E, BM, args.n_tiles_n);
        if (static_cast<int32_t>(pair) >= T) return;
    }

    if (threadIdx.x == 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 2 * pair_epilogue_warps<kEpi>());
        }
        mbar_init(drain_bar, 1);
        if constexpr (kDyn) {
            // q_empty (used in the leader) counts the leader's MMA thread and
            // epilogue warps and the peer's producer and epilogue warps
            for (int i = 0; i < kQueueDepth; ++i) {
                mbar_init(qfull_bar(i), 1);
                mbar_init(qempty_bar(i), 2 + 2 * pair_epilogue_warps<kEpi>());
            }
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmap_x);
        tma_prefetch_map(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&misc[0]), Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after_sync();

    const uint32_t tmem_base = misc[0];
    volatile uint32_t* abort_flag = &misc[1];
    const uint32_t peer_flag = map_to_rank(smem_addr(&misc[1]), rank ^ 1u);
    const int KB = args.num_k_blocks;
    const int nN = args.n_tiles_n;
    const int WO = args.walk_order;  // walk position t visits tile walk_tile(t, ...), the same in both CTAs
    const int32_t WS = walk_stride_for(T);
    auto tile_at = [&](int32_t p) -> TileCoord {
        return walk_decode(s_off, s_pre, s_order, s_spre, E, BM, kOutN, nN, T, WO, WS, p);
    };
    // Mixed launch: take the next descriptor from this CTA's queue and
    // release the slot on the leader's q_empty (`warp_wide`: all lanes of an
    // epilogue warp wait, lane 0 releases).  False on an abort.
    auto q_pop = [&](int& qs, uint32_t& qp, TileCoord& c, bool warp_wide) -> bool {
        bool ok = pair_wait_or_abort<true>(qfull_bar(qs), qp, abort_flag, peer_flag, args.status, args.timeout_ns);
        if (warp_wide) ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        const volatile int32_t* d = q_desc + 4 * qs;
        c.expert = d[0];
        c.row0 = d[1];
        c.rows = d[2];
        c.col0 = d[3];
        if (warp_wide) __syncwarp();
        if (!warp_wide || lane == 0) {
            if (rank == 0) mbar_arrive(qempty_bar(qs));
            else mbar_arrive_cluster(map_to_rank(qempty_bar(qs), 0));
        }
        if (++qs == kQueueDepth) {
            qs = 0;
            qp ^= 1u;
        }
        return true;
    };

    if (warp == 0) {
        // ---------------------------------------------------- S4: TMA producer
        if (lane == 0 && (args.debug_flags & kDebugProducerStall) == 0) {
            int st = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            uint32_t n_produced = 0;  // tiles loaded: the slot of the next one in the descriptor ring
            bool ok = true;
            auto produce = [&](const TileCoord& c) {
                (void)RGG_BOUNDS_OK(tile_ok(c.expert, c.row0, c.rows, c.col0, s_off, E, args.N), args.status);
                const bool half = half_tile(c);
                const int32_t a_row = c.row0 + (half ? 64 : 128) * static_cast<int32_t>(rank);
                const int ncols = pair_tile_cols<BN, kEpi>(c.col0, args.N);
                const int np = ncols / (2 * Cfg::kPanelN);  // panels this CTA loads
                // plain: this CTA's half of the tile's columns; SwiGLU: the gate (CTA 0) or up (CTA 1) columns
                const int32_t b_col = (kEpi == kEpiSwiGLU) ? c.col0 + (rank ? args.N : 0)
                                                           : c.col0 + (ncols / 2) * static_cast<int32_t>(rank);
                const CUtensorMap* xmap = half ? &tmap_x64 : &tmap_x;
                const uint32_t tx_bytes = 2u * ((half ? 64u : 128u) * 128u + np * Cfg::kPanelB);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!pair_wait_or_abort(empty_bar(st), ph ^ 1u, abort_flag, peer_flag, args.status,
                                            args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = map_to_rank(full_bar(st), 0);
                    if (rank == 0) {
                        // static walk: the MMA thread reads it after its wait on this stage (this
                        // arrive releases it)
                        if (!kDyn && kb == 0)
                            info_ring[n_produced++ % kInfoSlots] =
                                idesc_bf16_f32(half ? 128 : 256, pair_tile_cols<BN, kEpi>(c.col0, args.N), true);
                        mbar_arrive_expect_tx(full_bar(st), tx_bytes);
                    }
                    // the second CTA's rows may start past M_tot (a short tile at the end of X): the copy
                    // zero-fills them, so the row check allows one tile of overhang
                    if (RGG_BOUNDS_OK(x_box_ok(kb * Cfg::kKStage, a_row, args.K, args.M_tot + 128, 2), args.status))
                        tma_load_2d_pair(a0 + st * sp.a_stage, xmap, full_leader, kb * Cfg::kKStage, a_row);
#pragma unroll
                    for (int p = 0; p < Cfg::kPanels; ++p) {
                        // a gate-up tail tile: panel 0 this CTA's 64 gate columns, panel 1 their up columns
                        const int32_t wc = (kEpi == kEpiSwiGLU && half)
                                               ? (p == 0 ? c.col0 : args.N + c.col0) +
                                                     Cfg::kPanelN * static_cast<int32_t>(rank)
                                               : b_col + Cfg::kPanelN * p;
                        if (p < np && RGG_BOUNDS_OK(w_box_ok(wc, kb * Cfg::kKStage, c.expert,
                                                             kEpi == kEpiSwiGLU ? 2 * int64_t(args.N) : args.N,
                                                             args.K, E, 2, Cfg::kPanelN),
                                                    args.status))
                            tma_load_3d_pair(b0 + st * sp.b_stage + p * Cfg::kPanelB, &tmap_w, full_leader, wc,
                                             kb * Cfg::kKStage, c.expert);
                    }
                    ++issued;
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            };
            if (kDyn && !args.sched_claims) {
                ClassWalk cw;
                cw.init(L, true, single_units > 0);
                for (int32_t p = pair; ok && p < cw.n_positions; p += pair_units) produce(cw.at(L, p));
            } else if constexpr (kDyn) {
                int qs = 0;
                uint32_t qp = 0;
                if (rank == 0) {
                    // claim, write the descriptor into both CTAs' queues, load the leader's half
                    TileClaimer cl;
                    cl.init(args.sched, L, true, static_cast<int32_t>(pair), args.sched_pairs, args.sched_singles);
                    TileCoord c = cl.next(L);
                    while (ok) {
                        if (!pair_wait_or_abort<true>(qempty_bar(qs), qp ^ 1u, abort_flag, peer_flag, args.status,
                                                      args.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        int32_t* d = q_desc + 4 * qs;
                        d[0] = c.expert;
                        d[1] = c.row0;
                        d[2] = c.rows;
                        d[3] = c.col0;
                        st_shared_cluster_v4(map_to_rank(smem_addr(d), 1), c.expert, c.row0, c.rows, c.col0);
                        mbar_arrive(qfull_bar(qs));
                        mbar_arrive_cluster(map_to_rank(qfull_bar(qs), 1));
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
                    TileCoord c;
                    while (ok) {
                        if (!q_pop(qs, qp, c, false)) {
                            ok = false;
                            break;
                        }
                        if (c.expert < 0) break;
                        produce(c);
                    }
                }
            } else {
                for (int32_t t = pair; ok && t < T; t += npairs) produce(tile_at(t));
            }
            if (!ok) {
                // The leader's full barriers count both CTAs' bytes: it waits
                // for the stages it armed; the peer gives its copies a grace
                // period (they land in microseconds).
                if (rank == 0) {
                    const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
                    for (uint32_t i = issued - n; i < issued; ++i)
                        wait_bounded(full_bar(static_cast<int>(i % S)), (i / S) & 1u, kDrainLimitNs);
                } else {
                    spin_ns(200000ull);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- S5: MMA issuer (leader only)
        if (lane == 0 && rank == 0) {
            int st = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true;
            uint32_t n_tiles = 0;  // tiles issued: the slot of the next one in the producer's descriptor ring
            // One tile.  from_ring (the static walk): its instruction
            // descriptor is the producer's ring entry, read once the tile's
            // first stage has landed; else `idesc`, decoded here.
            auto mma_tile = [&](uint32_t idesc, bool from_ring) {
                if (!pair_wait_or_abort(acce_bar(acc), acc_ph ^ 1u, abort_flag, peer_flag, args.status,
                                        args.timeout_ns)) {
                    ok = false;
                    return;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!pair_wait_or_abort(full_bar(st), ph, abort_flag, peer_flag, args.status, args.timeout_ns)) {
                        ok = false;
                        return;
                    }
                    tc_fence_after_sync();
                    if (kb == 0 && from_ring) idesc = info_ring[n_tiles % kInfoSlots];
                    const uint32_t a_st = a0 + st * sp.a_stage;
                    const uint32_t b_st = b0 + st * sp.b_stage;
#pragma unroll
                    for (int j = 0; j < kMmasPerStage; ++j) {
                        const uint64_t ad = sw128_desc(a_st + 32u * j, 16u, 1024u);
                        const uint64_t bd = sw128_desc(b_st + Cfg::kBStep * j, Cfg::kPanelB, 1024u);
                        mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair(empty_bar(st), 0x3);
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit_pair(accf_bar(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_ph ^= 1u;
                }
                ++n_tiles;
            };
            if (kDyn && !args.sched_claims) {
                ClassWalk cw;
                cw.init(L, true, single_units > 0);
                for (int32_t p = pair; ok && p < cw.n_positions; p += pair_units) {
                    const TileCoord c = cw.at(L, p);
                    mma_tile(idesc_bf16_f32(half_tile(c) ? 128 : 256, pair_tile_cols<BN, kEpi>(c.col0, args.N), true),
                             false);
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
                    mma_tile(idesc_bf16_f32(half_tile(c) ? 128 : 256, pair_tile_cols<BN, kEpi>(c.col0, args.N), true),
                             false);
                }
            } else {
                // every position of the walk is a tile: count them, take the descriptors from the ring
                const int32_t b = static_cast<int32_t>(pair);  // < T: the others left after S1
                const int32_t count = (T - b + static_cast<int32_t>(npairs) - 1) / static_cast<int32_t>(npairs);
                for (int32_t i = 0; ok && i < count; ++i) mma_tile(0u, true);
            }
            if (!ok) {
                mma_commit_pair(drain_bar, 0x1);
                wait_bounded(drain_bar, 0u, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- S6: epilogue
        const int q = warp & 3;
        const int N = args.N;
        int acc = 0;
        uint32_t acc_ph = 0;
        // false when the pair aborts
        auto epi_tile = [&](const TileCoord& c) -> bool {
            bool ok = pair_wait_or_abort(accf_bar(acc), acc_ph, abort_flag, peer_flag, args.status, args.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) return false;
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            // M = 256: this CTA's 128 rows, one per TMEM lane, all BN columns.
            // M = 128: this CTA's 64 rows fill the 128 lanes twice over (GB300
            // layout, probed with one-hot operands): lane L < 64 holds row L,
            // columns [0, BN/2); lane 64 + L holds row L, columns [BN/2, BN);
            // both in TMEM columns [0, BN/2).
            const bool half = half_tile(c);
            const int r_local = half ? 64 * static_cast<int>(rank) + 32 * (q & 1) + lane
                                     : 128 * static_cast<int>(rank) + q * 32 + lane;
            const int tcols = (kEpi == kEpiSwiGLU) ? kOutN : pair_tile_cols<BN, kEpi>(c.col0, N);
            const int ncols = half ? tcols / 2 : tcols;
            const int cbase = half ? (q >> 1) * (tcols / 2) : 0;  // first tile column this warp holds
            const bool row_ok = r_local < c.rows;
            const int64_t row = static_cast<int64_t>(c.row0) + r_local;
            const int32_t row_lo = s_off[c.expert], row_hi = s_off[c.expert + 1];  // the debug build's row bounds
            (void)row_lo;
            (void)row_hi;
            __nv_bfloat16* yrow = args.Y + row * N + c.col0 + cbase;
            constexpr int kParts = pair_epilogue_warps<kEpi>() / 4;  // warps per lane quadrant
            const int pc = ncols / kParts;                                // columns each of them writes
            const int c0 = ((warp - 2) >> 2) * pc;
#pragma unroll 1
            for (int cc = c0; cc < c0 + pc; cc += 32) {
                if (c.col0 + cbase + cc >= N) break;  // columns past N: not computed, not stored
                uint32_t v[32];
                const uint32_t tcol = static_cast<uint32_t>(acc * BN + cc);
                const bool ld_ok = RGG_BOUNDS_OK(tmem_cols_ok(tcol, 32, Cfg::kTmemCols), args.status);
                if (ld_ok) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(cc), v);
                if constexpr (kEpi == kEpiSwiGLU) {
                    // gate in columns [cc, cc+32), up in [up_off + cc, up_off + cc + 32): kOutN
                    // columns on (M = 256), half that on an M = 128 tail tile
                    const int up_off = half ? kOutN / 2 : kOutN;
                    uint32_t u[32];
                    const bool ldu_ok = RGG_BOUNDS_OK(tmem_cols_ok(tcol + up_off, 32, Cfg::kTmemCols), args.status);
                    if (ldu_ok) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(up_off + cc), u);
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
                if (row_ok) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = c.col0 + cbase + cc + 16 * h;
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
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar(acc), 0));
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1u;
            }
            return true;
        };
        if (kDyn && !args.sched_claims) {
            ClassWalk cw;
            cw.init(L, true, single_units > 0);
            for (int32_t p = pair; p < cw.n_positions; p += pair_units)
                if (!epi_tile(cw.at(L, p))) break;
        } else if constexpr (kDyn) {
            int qs = 0;
            uint32_t qp = 0;
            TileCoord c;
            while (q_pop(qs, qp, c, true) && c.expert >= 0)
                if (!epi_tile(c)) break;
        } else {
            for (int32_t t = pair; t < T; t += npairs)
                if (!epi_tile(tile_at(t))) break;
        }
    }

    tc_fence_before_sync();
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
    if constexpr (kDyn)
        if (threadIdx.x == 0 && args.sched_claims) sched_cta_done(args.sched, args.sched_total);  // after the leader's last claim
}

}  // namespace rgg
