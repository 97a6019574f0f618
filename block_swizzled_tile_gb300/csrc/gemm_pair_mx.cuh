// Persistent CTA-pair MXFP8 GEMM (tcgen05.mma cta_group::2, kind::mxf8f6f4
// with E8M0 block scales, scale_vec::1X) for sm_103a.
//
// The MXFP8 workload of "MI450 WMMA and ds_load Scheduling via a DAG
// Mutation" ("An example run on a real kernel": float8 e4m3 A and B with one
// power-of-two scale per 32 K elements of every row of A and column of B) on
// 256 x BN output tiles, ordered by the GemmIdentityBlockSwizzle map of
// "Block Scheduler Code Explained" (sections 4-7).  As in gemm_pair_kernel,
// the two CTAs of a cluster share a tile: the leader (rank 0) holds A rows
// 0-127 and B columns [0, BN/2) of every k-block, the peer A rows 128-255 and
// B columns [BN/2, BN); one thread of the leader issues the MMAs for both.
// A tile needs no split of K, so no partial sums cross the pair.
//
// Scale factors.  Each CTA's tensor memory must hold the A scales of its own
// 128 rows and the B scales of all BN columns, in the line order that
// tcgen05.cp 32x128b.warpx4 copies (16-byte line l = rows l, l+32, l+64,
// l+96, 4 bytes each: the codes of a k-block's four 32-element blocks).  The
// codes arrive by TMA, 32 bytes (8 k-blocks) per row per group, issued by the
// A-load thread in line with its k-blocks, two groups ahead: the first groups
// go out ahead of every operand tile, and no other role waits for room in
// the TMA queue the operand tiles keep full.  (Ordinary loads of rows 16 bytes
// apart are no alternative: with almost all of the SM's L1 given to shared
// memory they complete about one cache line per tens of nanoseconds.)  A
// scale warp in each CTA rewrites a group into line order in one slot of a
// two-group scale ring in its own shared memory, fences it for the async
// proxy and arrives on the leader's sf_full barrier of that slot (the peer
// after a release fence at cluster scope restricted to shared memory, with a
// relaxed arrival).  The leader's MMA warp waits there
// (acquire at cluster scope) once per group, then per k-block
// copies the lines of both CTAs into their tensor memories with one
// tcgen05.cp.cta_group::2 per 128 rows and issues the four MMAs.  The commit
// after a group's last k-block frees the slot in both CTAs (sf_empty).  One
// cross-CTA handshake per 8 k-blocks, not per k-block.
//
// Warps (256 threads): 0 lane 0 A loads (the leader's is the one arrival on
// full[], expecting both CTAs' bytes), 1 MMA (leader; whole warp waits, lane
// 0 issues), 2-5 epilogue (both CTAs), 6 lane 0 B loads, 7 scale factors.
// Two TMEM accumulators for 128-column tiles (the epilogue of one tile
// overlaps the next tile's MMAs), one for 256-column tiles.
#pragma once
#include "gemm_pair.cuh"

namespace bst {

constexpr uint32_t kPairMxThreads = 256;
constexpr uint32_t kPairMxScaleWarp = 7;
constexpr uint32_t kGroupKb = 8;            // k-blocks per scale group (one cross-CTA handshake each)
constexpr uint32_t kSfGroups = 2;           // slots of the scale ring
constexpr uint32_t kRawSlots = 3;           // raw code groups by TMA, issued two groups ahead

template <uint32_t BN, uint32_t STAGES>
struct PairMxLayout {
    static constexpr uint32_t ACC = BN == 128 ? 2u : 1u;
    static constexpr uint32_t kABytes = kBM * kLine;             // 128 A rows x 128 e4m3
    static constexpr uint32_t kBBytes = (BN / 2) * kLine;        // BN/2 B rows x 128 e4m3
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kSfaKb = 32 * 16;                  // a k-block's lines of the CTA's 128 A rows
    static constexpr uint32_t kSfbKb = BN * 4;                   // ... of all BN B columns
    static constexpr uint32_t kSfKb = kSfaKb + kSfbKb;
    static constexpr uint32_t kSfSlotBytes = kGroupKb * kSfKb;   // one group of k-blocks
    static constexpr uint32_t kSfOff = STAGES * kStageBytes;
    // raw codes as TMA delivers them: 4 bytes per k-block, kGroupKb k-blocks
    // per row, the CTA's 128 A rows then the tile's BN B columns
    static constexpr uint32_t kRawRow = 4 * kGroupKb;
    static constexpr uint32_t kRawA = kBM * kRawRow;
    static constexpr uint32_t kRawSlotBytes = (kBM + BN) * kRawRow;
    static constexpr uint32_t kRawOff = kSfOff + kSfGroups * kSfSlotBytes;
    static constexpr uint32_t kEpiOff = kRawOff + kRawSlots * kRawSlotBytes;
    static constexpr uint32_t kBarOff = kEpiOff + 4 * kEpiWarpBytes;
    // full, empty [STAGES]; tfull, tempty [ACC]; sf_full, sf_empty [kSfGroups]; drain;
    // raw_full, raw_empty [kRawSlots]; last
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * ACC + 2 * kSfGroups + 1 + 2 * kRawSlots + 1;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    // TMEM: ACC accumulators of BN columns, then scale factors of kGroupKb *
    // kSfGroups k-blocks (4 columns of A codes and BN / 32 of B codes each)
    static constexpr uint32_t kSfCols = 4 + BN / 32;
    static constexpr uint32_t kSfSlots = kGroupKb * kSfGroups;
    static constexpr uint32_t kColsUsed = ACC * BN + kSfSlots * kSfCols;
    static constexpr uint32_t kTmemCols = kColsUsed <= 256 ? 256 : 512;
    static_assert(kColsUsed <= 512, "TMEM budget");
    static_assert(kStageBytes % 1024 == 0 && kSfSlotBytes % 1024 == 0, "1024-byte alignment of the ring");
    static constexpr uint32_t smem_bytes() { return 1024 + kMiscOff + 16; }
};

// L2 prefetch of the scale codes a CTA of the pair reads for one tile: its
// 128 rows of A's codes and the tile's BN columns of B's (K/32 bytes each),
// spread over `nthreads` threads.  Every address is a byte that exists.
template <uint32_t BN>
__device__ __forceinline__ void prefetch_scale_rows(const GemmArgs& g, const TileInfo& ti, uint32_t rank,
                                                    uint32_t tid, uint32_t nthreads) {
    const uint32_t lines_per_row = (g.sf_ld + 127) / 128;
    for (uint32_t L = tid; L < (kBM + BN) * lines_per_row; L += nthreads) {
        const uint32_t r = L / lines_per_row, c = (L % lines_per_row) * 128;
        const bool is_a = r < kBM;
        const uint32_t row = is_a ? ti.row0 + rank * kBM + r : ti.n * BN + (r - kBM);
        if (row < (is_a ? g.M : g.N)) prefetch_l2((is_a ? g.sfa : g.sfb) + static_cast<int64_t>(row) * g.sf_ld + c);
    }
}

template <uint32_t BN, uint32_t STAGES>
__global__ void __launch_bounds__(kPairMxThreads, 1) gemm_pair_mx_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = PairMxLayout<BN, STAGES>;
    static_assert(BN == 128 || BN == 256, "BN");
    constexpr uint32_t ACC = Lay::ACC;
    constexpr uint32_t TM = 2 * kBM;
    constexpr uint32_t BH = BN / 2;
    constexpr uint32_t bk_elems = 128;               // e4m3: 128 per 128-byte line
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m, &prm.g.ps};
    const uint32_t num_kb = prm.g.num_kb;            // a multiple of kGroupKb (K a multiple of 1024)
    const uint32_t total_tiles = prm.g.total_tiles;
    uint32_t* const err = prm.g.err;
    uint64_t* const tl = prm.g.timeline ? prm.g.timeline + static_cast<uint64_t>(blockIdx.x) * 64 : nullptr;
    const uint64_t t_entry = globaltimer_ns();

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + ACC;
    uint64_t* sf_full = tempty + ACC;
    uint64_t* sf_empty = sf_full + kSfGroups;
    uint64_t* drain = sf_empty + kSfGroups;
    uint64_t* raw_full = drain + 1;
    uint64_t* raw_empty = raw_full + kRawSlots;
    uint64_t* last = raw_empty + kRawSlots;          // single use: the CTA's last tile is accumulated
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();            // 0 leader, 1 peer
    const uint32_t cid = cluster_id_x();
    const uint32_t nclusters = num_clusters_x();
    const GroupTable gt{nullptr, nullptr, 0};

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (uint32_t a = 0; a < ACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);                // one arrival per epilogue warp of both CTAs
        }
        for (uint32_t g = 0; g < kSfGroups; ++g) {
            mbar_init(&sf_full[g], 2);               // the scale warps of both CTAs (the leader's is used)
            mbar_init(&sf_empty[g], 1);
        }
        mbar_init(drain, 1);
        for (uint32_t r = 0; r < kRawSlots; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], 1);
        }
        mbar_init(last, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&prm.tmap_a);
        prefetch_tmap(&prm.tmap_b);
        prefetch_tmap(&prm.tmap_sfa);
        prefetch_tmap(&prm.tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Lay::kTmemCols);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                  // barriers of both CTAs initialised
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    // the first tile's coordinates come from the arguments alone
    const TileInfo ti0 = cid < total_tiles ? tile_info(sa, cid, TM, BN, gt) : TileInfo{};
    if (cid < total_tiles && warp >= 2 && warp < 6) {
        // the epilogue warps pull the first tile's scale codes into L2 while
        // the previous kernel finishes (a prefetch reads nothing into the SM)
        prefetch_scale_rows<BN>(prm.g, ti0, rank, threadIdx.x - 64, 128);
    }
    griddep_wait();
    if (tl && threadIdx.x == 0) tl[53] = globaltimer_ns();
    griddep_launch_dependents();
    if (tl && threadIdx.x == 0) { tl[0] = t_entry; tl[52] = globaltimer_ns(); }

    if ((warp == 0 || warp == kPairBWarp) && lane == 0) {
        // ------------------------------------------------------ producer --
        const bool is_a = warp == 0;
        const uint32_t full_leader = map_to_cta(smem_u32(full), 0);
        constexpr uint32_t tx = Lay::kABytes + Lay::kBBytes;
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        // The A thread also loads this CTA's scale codes by TMA, a raw group
        // (kGroupKb k-blocks) at a time, kRawSlots - 1 groups ahead of the
        // k-block it issues: one thread feeds the TMA queue in order, so no
        // other role waits behind a full queue (group 0 alone is issued by the
        // scale warp, before any operand tile is queued).  A raw slot is
        // refilled once the scale warp has read it (raw_empty).
        const uint32_t ngroups = num_kb / kGroupKb;
        const uint32_t my_tiles = cid < total_tiles ? (total_tiles - cid + nclusters - 1) / nclusters : 0u;
        const uint32_t total_groups = my_tiles * ngroups;
        uint32_t rg = total_groups ? 1u : 0u;        // raw groups issued (group 0 by the scale warp)
        TileInfo ti_issue = ti0;
        uint32_t t_issue = cid;
        auto issue_raw = [&]() -> bool {
            const uint32_t G = rg, r = G % kRawSlots;
            if (G >= kRawSlots && !mbar_wait(&raw_empty[r], ((G / kRawSlots) & 1u) ^ 1u, ctl, 12)) return false;
            const uint32_t tile = cid + (G / ngroups) * nclusters;
            if (tile != t_issue) { ti_issue = tile_info(sa, tile, TM, BN, gt); t_issue = tile; }
            uint8_t* slot = smem + Lay::kRawOff + r * Lay::kRawSlotBytes;
            mbar_arrive_expect_tx(&raw_full[r], Lay::kRawSlotBytes);
            const int32_t x = static_cast<int32_t>((G % ngroups) * Lay::kRawRow);
            tma_load_2d(slot, &prm.tmap_sfa, &raw_full[r], x, static_cast<int32_t>(ti_issue.row0 + rank * kBM));
            tma_load_2d(slot + Lay::kRawA, &prm.tmap_sfb, &raw_full[r], x, static_cast<int32_t>(ti_issue.n * BN));
            ++rg;
            return true;
        };
        // the next groups after k-blocks 0, 8, 16, ... (each about two groups
        // ahead of the MMAs)
        if (tl && is_a) tl[54] = globaltimer_ns();
        for (uint32_t t = cid; ok && t < total_tiles; t += nclusters) {
            const TileInfo ti = t == cid ? ti0 : tile_info(sa, t, TM, BN, gt);
            const int32_t row = is_a ? static_cast<int32_t>(ti.row0 + rank * kBM)
                                     : static_cast<int32_t>(ti.n * BN + rank * BH);
            const uint32_t dst_off = is_a ? 0u : Lay::kABytes;
            const CUtensorMap* map = is_a ? &prm.tmap_a : &prm.tmap_b;
            for (uint32_t kb = 0; kb < num_kb; ++kb) {
                // the ring starts empty: only a stage being reused is waited for
                if (issued >= STAGES && !mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                uint8_t* st = smem + stage * Lay::kStageBytes;
                if (is_a && rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                tma_load_2d_pair(st + dst_off, map, full_leader + stage * 8, static_cast<int32_t>(kb * bk_elems), row);
                if (tl && is_a && issued < 15) tl[1 + issued] = globaltimer_ns();
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (is_a && kb % kGroupKb == 0 && rg < total_groups && !issue_raw()) { ok = false; break; }
            }
        }
        if (!ok && is_a) {
            // let the raw code copies in flight land before the CTA exits
            for (uint32_t G = rg >= kRawSlots ? rg - kRawSlots : 0u; G < rg; ++G)
                mbar_wait_drain(&raw_full[G % kRawSlots], (G / kRawSlots) & 1u, ctl.timeout_ns);
        }
        if (!ok && rank == 0 && is_a) {
            // let the copies of both CTAs already counted here land
            uint32_t s = stage, ph = phase;
            const uint32_t pending = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < pending; ++i) {
                if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
            }
        }
    } else if (warp == kPairMxScaleWarp) {
        // ------------------------------------------------- scale factors --
        // The CTA's groups of kGroupKb k-blocks, in order over its tiles: the
        // raw codes the A thread loaded into raw slot G % kRawSlots are
        // rewritten into line order in ring slot G % kSfGroups.
        const uint32_t sf_full_leader = map_to_cta(smem_u32(sf_full), 0);
        const uint32_t ngroups = num_kb / kGroupKb;
        const uint32_t my_tiles = cid < total_tiles ? (total_tiles - cid + nclusters - 1) / nclusters : 0u;
        const uint32_t total_groups = my_tiles * ngroups;
        if (lane == 0 && total_groups) {
            // group 0 goes out from here, in parallel with the A thread's
            // first operand tile
            uint8_t* slot = smem + Lay::kRawOff;
            mbar_arrive_expect_tx(&raw_full[0], Lay::kRawSlotBytes);
            tma_load_2d(slot, &prm.tmap_sfa, &raw_full[0], 0, static_cast<int32_t>(ti0.row0 + rank * kBM));
            tma_load_2d(slot + Lay::kRawA, &prm.tmap_sfb, &raw_full[0], 0, static_cast<int32_t>(ti0.n * BN));
        }
        __syncwarp();
        for (uint32_t G = 0; G < total_groups; ++G) {
            if (!warp_wait(&raw_full[G % kRawSlots], (G / kRawSlots) & 1u, ctl, 6)) break;
            const uint32_t slot = G % kSfGroups, ph = (G / kSfGroups) & 1u;
            if (!warp_wait(&sf_empty[slot], ph ^ 1u, ctl, 7)) break;
            // lane l: rows l, l+32, l+64, l+96 of A's codes and of each 128 B
            // columns, 32 bytes (8 k-blocks) each, read as two 16-byte words
            const uint8_t* raw = smem + Lay::kRawOff + (G % kRawSlots) * Lay::kRawSlotBytes + lane * Lay::kRawRow;
            constexpr uint32_t kRows = 4 * (1 + BN / 128);
            uint4 rr[kRows][2];
#pragma unroll
            for (uint32_t i = 0; i < kRows; ++i) {
                const uint4* src = reinterpret_cast<const uint4*>(raw + i * 32 * Lay::kRawRow);
                rr[i][0] = src[0];
                rr[i][1] = src[1];
            }
            auto word = [&](uint32_t i, uint32_t j) {
                const uint4& h = rr[i][j >> 2];
                const uint32_t w = j & 3u;
                return w == 0 ? h.x : w == 1 ? h.y : w == 2 ? h.z : h.w;
            };
            uint8_t* lines = smem + Lay::kSfOff + slot * Lay::kSfSlotBytes + lane * 16u;
#pragma unroll
            for (uint32_t j = 0; j < kGroupKb; ++j) {
                uint8_t* kbl = lines + j * Lay::kSfKb;
                *reinterpret_cast<uint4*>(kbl) = make_uint4(word(0, j), word(1, j), word(2, j), word(3, j));
#pragma unroll
                for (uint32_t h = 0; h < BN / 128; ++h)
                    *reinterpret_cast<uint4*>(kbl + Lay::kSfaKb + h * 512u) =
                        make_uint4(word(4 + 4 * h, j), word(5 + 4 * h, j), word(6 + 4 * h, j), word(7 + 4 * h, j));
            }
            // generic writes -> the leader's tcgen05.cp reads, and the raw
            // slot's generic reads -> its next TMA write
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&raw_empty[G % kRawSlots]);
                if (rank == 0) {
                    mbar_arrive(&sf_full[slot]);
                } else {
                    // the lines are this CTA's shared memory: a release
                    // restricted to it, then a relaxed arrival on the leader
                    fence_release_smem_cluster();
                    mbar_arrive_cluster_relaxed(sf_full_leader + slot * 8);
                }
            }
            if (tl && lane == 0 && G < 6) tl[56 + G] = globaltimer_ns();
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (leader) --
        if (rank == 0) {
            const uint32_t smem_base = smem_u32(smem);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, gi = 0, kbg = 0;
            bool ok = true, any_mma = false;
            for (uint32_t t = cid; ok && t < total_tiles; t += nclusters) {
                if (!warp_wait(&tempty[acc], acc_phase ^ 1u, ctl, 2)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = 0; kb < num_kb; ++kb) {
                    const uint32_t j = kb % kGroupKb, slot = gi % kSfGroups;
                    if (j == 0) {
                        // both CTAs' scale lines of this group are written
                        const bool got = mbar_wait_cluster(&sf_full[slot], (gi / kSfGroups) & 1u, ctl, 8);
                        if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
                    }
                    if (!warp_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
                        if (tl && kbg < 16) tl[16 + kbg] = globaltimer_ns();
                        const uint32_t sf_col = tmem_base + ACC * BN + (kbg % Lay::kSfSlots) * Lay::kSfCols;
                        const uint32_t lines = smem_base + Lay::kSfOff + slot * Lay::kSfSlotBytes + j * Lay::kSfKb;
                        tmem_cp_32x128b_warpx4_pair(sf_col, smem_desc(lines, 0, 128, kSwizzleNone));
#pragma unroll
                        for (uint32_t h = 0; h < BN / 128; ++h)
                            tmem_cp_32x128b_warpx4_pair(sf_col + 4 + 4 * h,
                                                        smem_desc(lines + Lay::kSfaKb + h * 512, 0, 128, kSwizzleNone));
                        const uint32_t sa_addr = smem_base + stage * Lay::kStageBytes;
                        const uint64_t adesc = smem_desc(sa_addr, 16, 1024, kSwizzle128B);
                        const uint64_t bdesc = smem_desc(sa_addr + Lay::kABytes, 16, 1024, kSwizzle128B);
#pragma unroll
                        for (uint32_t kk = 0; kk < 4; ++kk)
                            umma_mxf8_pair(d_tmem, adesc + ((kk * 32u) >> 4), bdesc + ((kk * 32u) >> 4),
                                           idesc_mxf8(TM, BN, kk), sf_col, sf_col + 4,
                                           (kb > 0 || kk > 0) ? 1u : 0u);
                        umma_commit_pair_mc(&empty[stage], 0x3);
                        if (j == kGroupKb - 1) umma_commit_pair_mc(&sf_empty[slot], 0x3);
                    }
                    __syncwarp();
                    any_mma = true;
                    ++kbg;
                    if (j == kGroupKb - 1) ++gi;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (elect_one()) {
                    umma_commit_pair_mc(&tfull[acc], 0x3);
                    // after the last tile also the single-use barrier (a parity
                    // wait on tfull could match an earlier phase)
                    if (t + nclusters >= total_tiles) umma_commit_pair_mc(last, 0x3);
                }
                __syncwarp();
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (lane == 0 && !ok && any_mma) {
                // every tcgen05 op issued so far must finish before TMEM is freed
                umma_commit_pair_mc(drain, 0x1);
                mbar_wait_drain(drain, 0, ctl.timeout_ns);
            }
        }
    }

    // ----------------------------------------------------- epilogue (both) --
    // Warps 2-5 finish every tile (TMEM lane quarter warp % 4).  For the
    // CTA's last tile, warps 0, 1, 6 and 7 -- one per lane quarter, idle once
    // their loads, MMAs and scale codes are issued -- take columns [BN/2, BN)
    // and stage their stores in the ring, which is idle by then.
    const uint32_t my_tiles = cid < total_tiles ? (total_tiles - cid + nclusters - 1) / nclusters : 0u;
    const bool main_epi = warp >= 2 && warp < 6;
    __syncwarp();                                    // reconverge the single-lane roles
    if (my_tiles && (main_epi || warp < 2 || warp >= kPairBWarp)) {
        const uint32_t q = warp & 3u;                    // TMEM lane quarter of this warp
        const uint32_t wrow = rank * kBM + q * 32;       // first row of this warp in the 256-row tile
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
        uint8_t* const epi_stage = smem + (main_epi ? Lay::kEpiOff : 0u) + q * kEpiWarpBytes;
        const int64_t ldc = prm.g.ldc;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        const uint32_t tempty_leader = map_to_cta(smem_u32(tempty), 0);
        // columns [c0, c1) of a tile's accumulator acc of this warp's 32 rows
        auto finish = [&](const TileInfo& ti, uint32_t acc, uint32_t c0, uint32_t c1) {
            const uint32_t rows_valid = ti.m_act > wrow ? min(32u, ti.m_act - wrow) : 0u;   // warp-uniform
            uint8_t* const cwarp = prm.g.C + static_cast<int64_t>(ti.row0 + wrow) * ldc * csize;
            const uint32_t taddr = tmem_base + ((q * 32) << 16) + acc * BN;
#pragma unroll 1
            for (uint32_t cc = c0 / 32; cc < c1 / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + cc * 32, v);
                if (rows_valid && cc * 32 < ti.n_act)
                    store_chunk_coalesced(epi_stage, c_type, c_vec,
                                          cwarp + static_cast<int64_t>(ti.n * BN + cc * 32) * csize, ldc * csize,
                                          rows_valid, min(32u, ti.n_act - cc * 32), v, lane);
            }
        };
        if (main_epi) {
            uint32_t acc = 0, acc_phase = 0, ep_tile = 0;
            for (uint32_t i = 0; i < my_tiles; ++i) {
                const uint32_t t = cid + i * nclusters;
                const TileInfo ti = i == 0 ? ti0 : tile_info(sa, t, TM, BN, gt);
                if (prm.g.trace && rank == 0 && warp == 2 && lane == 0 && t < prm.g.trace_cap) {
                    uint32_t* tr = prm.g.trace + static_cast<uint64_t>(t) * 5;
                    tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
                }
                if (!warp_wait(&tfull[acc], acc_phase, ctl, 4)) break;
                tc_fence_after();
                if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[32 + ep_tile] = globaltimer_ns();
                finish(ti, acc, 0, i + 1 == my_tiles ? BN / 2 : BN);
                // the accumulator's reads are complete (tcgen05.wait::ld): a
                // relaxed arrival releases it, with no data to publish
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
                if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[40 + ep_tile] = globaltimer_ns();
                ++ep_tile;
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
        } else {
            // the last tile's accumulator: tile index my_tiles - 1, complete
            // once the single-use barrier `last` has fired
            const uint32_t i = my_tiles - 1;
            const uint32_t acc = i % ACC;
            const TileInfo ti = i == 0 ? ti0 : tile_info(sa, cid + i * nclusters, TM, BN, gt);
            if (warp_wait(last, 0, ctl, 13)) {
                tc_fence_after();
                finish(ti, acc, BN / 2, BN);
            }
        }
    }

    if (tl && lane == 0 && warp <= 2) tl[48 + warp] = globaltimer_ns();
    // single-lane roles leave their warps diverged: reconverge every warp
    // first, so that the barrier counts each warp once; the cluster barrier
    // (with release: the epilogue's last arrivals on the leader's barriers
    // must land before the leader may leave) also orders this CTA's own warps
    // before TMEM is freed
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Lay::kTmemCols);
    }
}

}  // namespace bst
