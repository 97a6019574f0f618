// Persistent CTA-pair tcgen05 GEMM (cta_group::2) for sm_103a, fp16/bf16.
//
// Clusters of two CTAs on the two SMs of a TPC work together on output tiles
// of 256 x BN: the leader CTA (cluster rank 0) holds A rows 0-127 and B
// columns [0, BN/2) of each k-block in its shared memory, the peer (rank 1)
// holds A rows 128-255 and B columns [BN/2, BN).  One thread of the leader
// issues tcgen05.mma.cta_group::2 (M = 256), which reads both CTAs' shared
// memory and writes accumulator rows 0-127 into the leader's TMEM and rows
// 128-255 into the peer's.  Each SM therefore receives 128 + BN/2 operand rows
// per k-block for 128 x BN outputs -- a third less than a single-CTA
// 128 x BN tile needs -- which is what lets the tensor pipe outrun the L2->SM
// bandwidth.  The tile order is the same GemmIdentityBlockSwizzle map, on
// 256-row tiles ("Block Scheduler Code Explained", sections 4-7).
//
// Synchronisation of the pair:
//   full[s]   leader only; the leader's producer arrives once, expecting
//             the bytes of both CTAs, and both CTAs' TMA loads complete_tx
//             there (a peer's bytes may land before the leader's expect_tx:
//             the transaction count may go negative meanwhile, and the
//             missing arrival keeps the phase open).  A cluster-scope arrive
//             per k-block from the peer would instead wait on the peer's
//             outstanding copies every time.
//   empty[s]  in both CTAs; the leader's MMA commit multicasts to both.
//   tfull[a]  in both CTAs; the leader's MMA commit multicasts to both.
//   tempty[a] leader only; one arrival per epilogue warp of both CTAs (8).
// A cluster barrier after set-up (barriers initialised before any remote
// arrive) and before exit (no CTA leaves while the other may still touch its
// shared memory) brackets the work.
#pragma once
#include "gemm_kernel.cuh"

namespace bst {

template <uint32_t BN, uint32_t STAGES>
struct PairLayout {
    static constexpr uint32_t kACC = 2;
    static constexpr uint32_t kABytes = kBM * kLine;            // 128 A rows per CTA
    static constexpr uint32_t kBBytes = (BN / 2) * kLine;       // BN/2 B rows per CTA
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kBarOff = STAGES * kStageBytes;
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * kACC + 1;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kTableOff = (kMiscOff + 16 + 15) & ~15u;
    static constexpr uint32_t kTmemCols = kACC * BN <= 256 ? 256 : 512;
    static_assert(kACC * BN <= 512, "TMEM budget");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static constexpr uint32_t smem_bytes(uint32_t groups) { return 1024 + kTableOff + 8 * (groups + 1); }
};

template <uint32_t BN, uint32_t STAGES>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_pair_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = PairLayout<BN, STAGES>;
    constexpr uint32_t ACC = Lay::kACC;
    constexpr uint32_t TM = 2 * kBM;
    constexpr uint32_t BH = BN / 2;                  // B columns held by each CTA
    static_assert(BN == 128 || BN == 256, "BN");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m};
    const uint32_t N = prm.g.N, mode = prm.g.mode, num_kb = prm.g.num_kb, G = prm.g.G;
    const uint32_t a_mn = prm.g.a.mn_major, b_mn = prm.g.b.mn_major;
    const uint32_t a_rank3 = prm.g.a.tma_rank == 3, b_rank3 = prm.g.b.tma_rank == 3;
    uint32_t* const err = prm.g.err;
    uint64_t* const tl = prm.g.timeline ? prm.g.timeline + static_cast<uint64_t>(blockIdx.x) * 64 : nullptr;
    constexpr uint32_t bk_elems = 64;                // 16-bit operands: 64 per 128-byte line

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + ACC;
    uint64_t* drain = bars + 2 * STAGES + 2 * ACC;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    uint32_t* tiles_smem = misc + 2;

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();            // 0 leader, 1 peer
    const uint32_t cid = cluster_id_x();
    const uint32_t nclusters = num_clusters_x();

    GroupTable gt;
    gt.G = G;
    gt.tile_off = reinterpret_cast<uint32_t*>(smem + Lay::kTableOff);
    gt.row_off = gt.tile_off + (mode == kModeGrouped ? G + 1 : 0);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (uint32_t a = 0; a < ACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *tiles_smem = prm.g.total_tiles;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&prm.tmap_a);
        prefetch_tmap(&prm.tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Lay::kTmemCols);
        tmem_relinquish_pair();
    }
    if (mode == kModeGrouped && warp == 2)
        build_group_table(gt, prm.g.group_m, G, N, TM, BN, sa.total_m, err, tiles_smem, lane);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t total_tiles = *tiles_smem;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    if (tl && threadIdx.x == 0) tl[0] = globaltimer_ns();

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        // both CTAs: own A half and own B half, counted on the leader's full[s]
        const uint32_t full_leader = map_to_cta(smem_u32(full), 0);
        constexpr uint32_t tx = Lay::kABytes + Lay::kBBytes;
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        // a single thread issues every load (cheaper per k-block than a
        // warp-wide loop with one active lane)
        for (uint32_t t = cid; lane == 0 && ok && t < total_tiles; t += nclusters) {
            const TileInfo ti = tile_info(sa, t, TM, BN, gt);
            const uint32_t a_row = ti.row0 + rank * kBM;
            const uint32_t b_col = ti.n * BN + rank * BH;
            const int32_t zc = static_cast<int32_t>(ti.tag);
            for (uint32_t kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                {
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    uint8_t* sb_s = sa_s + Lay::kABytes;
                    const uint32_t bar = full_leader + stage * 8;
                    const int32_t k0 = kb * bk_elems;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                    if (!a_mn) {
                        if (a_rank3) tma_load_3d_pair(sa_s, &prm.tmap_a, bar, k0, a_row, zc);
                        else tma_load_2d_pair(sa_s, &prm.tmap_a, bar, k0, a_row);
                    } else {
                        for (uint32_t j = 0; j < kBM / bk_elems; ++j) {
                            if (a_rank3) tma_load_3d_pair(sa_s + j * bk_elems * kLine, &prm.tmap_a, bar, a_row + j * bk_elems, k0, zc);
                            else tma_load_2d_pair(sa_s + j * bk_elems * kLine, &prm.tmap_a, bar, a_row + j * bk_elems, k0);
                        }
                    }
                    if (!b_mn) {
                        if (b_rank3) tma_load_3d_pair(sb_s, &prm.tmap_b, bar, k0, b_col, zc);
                        else tma_load_2d_pair(sb_s, &prm.tmap_b, bar, k0, b_col);
                    } else {
                        for (uint32_t j = 0; j < BH / bk_elems; ++j) {
                            if (b_rank3) tma_load_3d_pair(sb_s + j * bk_elems * kLine, &prm.tmap_b, bar, b_col + j * bk_elems, k0, zc);
                            else tma_load_2d_pair(sb_s + j * bk_elems * kLine, &prm.tmap_b, bar, b_col + j * bk_elems, k0);
                        }
                    }
                    if (tl && issued < 15) tl[1 + issued] = globaltimer_ns();
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (lane == 0 && !ok && rank == 0) {
            // let the copies of both CTAs already counted here land
            uint32_t s = stage, ph = phase;
            const uint32_t pending = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < pending; ++i) {
                if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (leader) --
        if (rank == 0) {
            const uint32_t a_lbo = a_mn ? bk_elems * kLine : 16u;
            const uint32_t b_lbo = b_mn ? bk_elems * kLine : 16u;
            const uint32_t a_step = a_mn ? 16u * kLine : 32u;
            const uint32_t b_step = b_mn ? 16u * kLine : 32u;
            const uint32_t idesc = idesc_f16(prm.g.ab_fmt, a_mn, b_mn, TM, BN);
            const uint32_t smem_base = smem_u32(smem);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, mma_kb = 0;
            bool ok = true, any_mma = false;
            for (uint32_t t = cid; lane == 0 && ok && t < total_tiles; t += nclusters) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ctl, 2)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
                    tc_fence_after();
                    {
                        if (tl && mma_kb < 16) tl[16 + mma_kb] = globaltimer_ns();
                        const uint32_t sa_addr = smem_base + stage * Lay::kStageBytes;
                        const uint64_t adesc = smem_desc(sa_addr, a_lbo, 1024, kSwizzle128B);
                        const uint64_t bdesc = smem_desc(sa_addr + Lay::kABytes, b_lbo, 1024, kSwizzle128B);
#pragma unroll
                        for (uint32_t kk = 0; kk < 4; ++kk)
                            umma_f16_pair(d_tmem, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4), idesc,
                                          (kb > 0 || kk > 0) ? 1u : 0u);
                        umma_commit_pair_mc(&empty[stage], 0x3);
                    }
                    ++mma_kb;
                    any_mma = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_mc(&tfull[acc], 0x3);
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (lane == 0 && !ok && any_mma) {
                // every tcgen05 op issued so far must finish before TMEM is freed
                umma_commit_pair_mc(drain, 0x1);
                mbar_wait_drain(drain, 0, ctl.timeout_ns);
            }
        }
    } else {
        // ---------------------------------------------- epilogue (both) --
        prefetch_operands(prm.g, threadIdx.x - 64, 128);
        const uint32_t q = warp & 3u;                    // TMEM lane quarter of this warp
        const uint32_t r = rank * kBM + q * 32 + lane;   // row of this thread in the 256-row tile
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
        uint8_t* const C = prm.g.C;
        const int64_t ldc = prm.g.ldc, c_bs = prm.g.c_batch_stride;
        uint32_t* const trace = prm.g.trace;
        const uint32_t trace_cap = prm.g.trace_cap;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        const uint32_t tempty_leader = map_to_cta(smem_u32(tempty), 0);
        uint32_t acc = 0, acc_phase = 0, ep_tile = 0;
        bool ok = true;
        for (uint32_t t = cid; ok && t < total_tiles; t += nclusters) {
            const TileInfo ti = tile_info(sa, t, TM, BN, gt);
            if (trace && rank == 0 && warp == 2 && lane == 0) {
                if (t < trace_cap) {
                    uint32_t* tr = trace + static_cast<uint64_t>(t) * 5;
                    tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
                } else {
                    atomicOr(&err[0], kErrTraceOverflow);
                }
            }
            const bool row_ok = r < ti.m_act;
            const uint32_t grow = ti.row0 + r;
            const int64_t cbase = mode == kModeBatched ? static_cast<int64_t>(ti.tag) * c_bs : 0;
            uint8_t* crow = C + (cbase + static_cast<int64_t>(grow) * ldc) * csize;
            const uint32_t n0 = ti.n * BN;
            if (!warp_wait(&tfull[acc], acc_phase, ctl, 4)) { ok = false; break; }
            tc_fence_after();
            if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[32 + ep_tile] = globaltimer_ns();
            const uint32_t taddr = tmem_base + ((q * 32) << 16) + acc * BN;
#pragma unroll 1
            for (uint32_t cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + cc * 32, v);
                if (row_ok && cc * 32 < ti.n_act)
                    store_row_chunk(c_type, c_vec, crow, n0 + cc * 32, ti.n_act - cc * 32, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);
            if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[40 + ep_tile] = globaltimer_ns();
            ++ep_tile;
            if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
        }
    }

    if (tl && lane == 0 && warp <= 2) tl[48 + warp] = globaltimer_ns();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Lay::kTmemCols);
    }
}

}  // namespace bst

namespace bst {

// Split-K variant for problems with fewer 256 x BN tiles than the GPU has
// CTA pairs ("09_split_matmul" of "Block Dispatch Policies" names split
// GEMMs; the split here is along K).  A cluster of 2*S CTAs owns one tile:
// CTA pair p (cluster ranks 2p, 2p+1) accumulates k-blocks
// [p*ceil(kb/S), (p+1)*ceil(kb/S)) of it exactly as gemm_pair_kernel does.
// The S partial tiles are then summed through distributed shared memory:
// each split finishes R = 128/S of the 128 accumulator rows its CTA holds.
// After a cluster barrier (every pipeline of the cluster drained, so the
// stage buffers can be reused), epilogue warp q of each CTA sends its 32
// accumulator rows to the CTA of split 32q/R on the same half of the tile
// (reduce-scatter); after a second barrier each CTA adds the S slots it
// received for its R rows, rounds once and stores them.  Nothing goes
// through global memory and no second kernel runs.
template <uint32_t BN, uint32_t STAGES, uint32_t S>
struct SplitLayout {
    using Pair = PairLayout<BN, STAGES>;
    static constexpr uint32_t kRows = kBM / S;                     // rows each split finishes
    static constexpr uint32_t kRowFloats = BN + 4;                 // padded: conflict-free 16-byte stores
    static constexpr uint32_t kSlotBytes = kRows * kRowFloats * 4; // the rows one split sends
    static_assert(S * kSlotBytes <= STAGES * Pair::kStageBytes, "receive slots reuse the stage buffers");
};

template <uint32_t BN, uint32_t STAGES, uint32_t S>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_pair_splitk_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = PairLayout<BN, STAGES>;
    using SL = SplitLayout<BN, STAGES, S>;
    constexpr uint32_t TM = 2 * kBM;
    constexpr uint32_t BH = BN / 2;
    static_assert(S == 2 || S == 4, "splits");
    static_assert(BN == 256, "split-K runs 256 x 256 tiles");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m};
    const uint32_t num_kb = prm.g.num_kb;
    const uint32_t a_mn = prm.g.a.mn_major, b_mn = prm.g.b.mn_major;
    uint32_t* const err = prm.g.err;
    constexpr uint32_t bk_elems = 64;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* drain = bars + 2 * STAGES + 2 * Lay::kACC;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    uint64_t* const tl = prm.g.timeline ? prm.g.timeline + static_cast<uint64_t>(blockIdx.x) * 64 : nullptr;
    if (tl && threadIdx.x == 0) tl[0] = globaltimer_ns();
    const uint32_t crank = cluster_rank();
    const uint32_t split = crank >> 1, half = crank & 1u, leader = crank & ~1u;
    const uint16_t pair_mask = static_cast<uint16_t>(3u << leader);
    const uint32_t t = cluster_id_x();               // one tile per cluster
    const bool has_tile = t < prm.g.total_tiles;
    // balanced ranges: sizes differ by at most one; a range is empty only
    // when there are fewer k-blocks than splits
    const uint32_t kb_begin = (split * num_kb) / S, kb_end = ((split + 1) * num_kb) / S;
    const bool has_k = kb_end > kb_begin;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&tfull[0], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&prm.tmap_a);
        prefetch_tmap(&prm.tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Lay::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (tl && threadIdx.x == 0) tl[1] = globaltimer_ns();
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    GroupTable gt{nullptr, nullptr, 0};
    TileInfo ti{};
    if (has_tile) ti = tile_info(sa, t, TM, BN, gt);

    if (warp == 0 && lane == 0 && has_tile) {
        // ------------------------------------------------------ producer --
        const uint32_t full_leader = map_to_cta(smem_u32(full), leader);
        constexpr uint32_t tx = Lay::kABytes + Lay::kBBytes;
        const uint32_t a_row = ti.row0 + half * kBM;
        const uint32_t b_col = ti.n * BN + half * BH;
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
            uint8_t* sa_s = smem + stage * Lay::kStageBytes;
            uint8_t* sb_s = sa_s + Lay::kABytes;
            const uint32_t bar = full_leader + stage * 8;
            const int32_t k0 = kb * bk_elems;
            if (half == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx);
            if (!a_mn) tma_load_2d_pair(sa_s, &prm.tmap_a, bar, k0, a_row);
            else
                for (uint32_t j = 0; j < kBM / bk_elems; ++j)
                    tma_load_2d_pair(sa_s + j * bk_elems * kLine, &prm.tmap_a, bar, a_row + j * bk_elems, k0);
            if (!b_mn) tma_load_2d_pair(sb_s, &prm.tmap_b, bar, k0, b_col);
            else
                for (uint32_t j = 0; j < BH / bk_elems; ++j)
                    tma_load_2d_pair(sb_s + j * bk_elems * kLine, &prm.tmap_b, bar, b_col + j * bk_elems, k0);
            if (tl && issued < 14) tl[2 + issued] = globaltimer_ns();
            ++issued;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok && half == 0) {
            uint32_t s = stage, ph = phase;
            const uint32_t pending = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < pending; ++i) {
                if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
            }
        }
    } else if (warp == 1 && lane == 0 && has_tile && has_k && half == 0) {
        // ------------------------------------- MMA issuer (pair leaders) --
        const uint32_t a_lbo = a_mn ? bk_elems * kLine : 16u;
        const uint32_t b_lbo = b_mn ? bk_elems * kLine : 16u;
        const uint32_t a_step = a_mn ? 16u * kLine : 32u;
        const uint32_t b_step = b_mn ? 16u * kLine : 32u;
        const uint32_t idesc = idesc_f16(prm.g.ab_fmt, a_mn, b_mn, TM, BN);
        const uint32_t smem_base = smem_u32(smem);
        uint32_t stage = 0, phase = 0;
        bool ok = true, any_mma = false;
        for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
            if (!mbar_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa_addr = smem_base + stage * Lay::kStageBytes;
            const uint64_t adesc = smem_desc(sa_addr, a_lbo, 1024, kSwizzle128B);
            const uint64_t bdesc = smem_desc(sa_addr + Lay::kABytes, b_lbo, 1024, kSwizzle128B);
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk)
                umma_f16_pair(tmem_base, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4), idesc,
                              (kb > kb_begin || kk > 0) ? 1u : 0u);
            umma_commit_pair_mc(&empty[stage], pair_mask);
            if (tl && kb - kb_begin < 16) tl[16 + kb - kb_begin] = globaltimer_ns();
            any_mma = true;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) umma_commit_pair_mc(&tfull[0], pair_mask);
        else if (any_mma) {
            umma_commit_pair_mc(drain, static_cast<uint16_t>(1u << crank));
            mbar_wait_drain(drain, 0, ctl.timeout_ns);
        }
    }

    // every role of every CTA of the cluster is done with the pipeline: the
    // epilogue waits for its accumulator first
    bool acc_ok = true;
    if (warp >= 2 && has_tile && has_k) acc_ok = warp_wait(&tfull[0], 0, ctl, 4);
    if (tl && warp == 2 && lane == 0) tl[32] = globaltimer_ns();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (tl && threadIdx.x == 64) tl[33] = globaltimer_ns();

    // reduce-scatter: warp q's 32 rows go to split 32q/R (same half), into
    // the slot of the sending split
    if (warp >= 2 && has_tile) {
        const uint32_t q = warp & 3u;
        const uint32_t dest = 2 * ((q * 32) / SL::kRows) + half;      // a rank of this cluster: < 2*S
        const uint32_t row_in_slot = (q * 32) % SL::kRows + lane;
        const uint32_t slot =
            map_to_cta(smem_u32(smem), dest) + split * SL::kSlotBytes + row_in_slot * SL::kRowFloats * 4;
        const bool have = acc_ok && has_k;            // an empty range sends zeros
        const uint32_t taddr = tmem_base + ((q * 32) << 16);
#pragma unroll 1
        for (uint32_t cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            if (have) tmem_ld_32x32b_x32(taddr + cc * 32, v);
#pragma unroll
            for (uint32_t j = 0; j < 32; j += 4) {
                if (have) st_cluster_v4(slot + (cc * 32 + j) * 4, v[j], v[j + 1], v[j + 2], v[j + 3]);
                else st_cluster_v4(slot + (cc * 32 + j) * 4, 0u, 0u, 0u, 0u);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tl && threadIdx.x == 64) tl[34] = globaltimer_ns();
    cluster_sync();
    if (tl && threadIdx.x == 64) tl[35] = globaltimer_ns();

    // sum the S slots for rows [split*R, split*R + R) of this half and store
    if (warp >= 2 && has_tile) {
        const uint32_t e = threadIdx.x - 64;             // 0..127: S threads per row
        const uint32_t row = e / S;                      // 0..R-1
        const uint32_t c0 = (e % S) * (BN / S);          // BN/S columns per thread
        const uint32_t r = half * kBM + split * SL::kRows + row;   // row within the 256-row tile
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        uint8_t* crow = prm.g.C + (static_cast<int64_t>(ti.row0 + r) * prm.g.ldc) * csize;
        const float* base = reinterpret_cast<const float*>(smem) + row * SL::kRowFloats + c0;
#pragma unroll 1
        for (uint32_t cc = 0; cc < BN / S; cc += 32) {
            uint32_t v[32];
#pragma unroll
            for (uint32_t j = 0; j < 32; ++j) {
                float acc = 0.f;
#pragma unroll
                for (uint32_t sidx = 0; sidx < S; ++sidx) acc += base[sidx * (SL::kSlotBytes / 4) + cc + j];
                v[j] = __float_as_uint(acc);
            }
            const uint32_t col = c0 + cc;
            if (r < ti.m_act && col < ti.n_act)
                store_row_chunk(c_type, c_vec, crow, ti.n * BN + col, ti.n_act - col, v);
        }
        if (prm.g.trace && split == 0 && half == 0 && e == 0 && t < prm.g.trace_cap) {
            uint32_t* tr = prm.g.trace + static_cast<uint64_t>(t) * 5;
            tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
        }
    }
    if (tl && threadIdx.x == 64) tl[36] = globaltimer_ns();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Lay::kTmemCols);
    }
    if (tl && threadIdx.x == 0) tl[37] = globaltimer_ns();
}

}  // namespace bst
