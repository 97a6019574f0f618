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
//   tempty[a] leader only; one arrival per epilogue warp of both CTAs (8),
//             relaxed: a warp arrives once its reads of the accumulator have
//             completed (tcgen05.wait::ld), and publishes no data with it.
// A cluster barrier after set-up (barriers initialised before any remote
// arrive) and before exit (no CTA leaves while the other may still touch its
// shared memory) brackets the work.
#pragma once
#include "gemm_kernel.cuh"

namespace bst {

// Warps of the CTA-pair kernels: 0 issues A loads (and the leader's arrival
// on full[]), 1 the MMA, 2-5 the epilogue, 6 issues B loads (one thread
// issues a TMA about every 0.1-0.15 us, so A and B get a thread each).
constexpr uint32_t kPairThreads = 224;
constexpr uint32_t kPairBWarp = 6;
// The int8 per-token-dequant variant keeps 128 int32 running sums per thread,
// so its 256-column tiles take two epilogue warps per TMEM lane quarter:
// warps 2-5 finish columns 0-127, warps 7-10 columns 128-255.
template <uint32_t EPI>
constexpr uint32_t pair_threads() { return EPI == kEpiDequant ? 352u : kPairThreads; }
template <uint32_t EPI>
constexpr uint32_t pair_epi_warps() { return EPI == kEpiDequant ? 8u : 4u; }

// Depth of the ring of cluster-launch-control responses (dynamic tasks).
constexpr uint32_t kClcDepth = 4;

// The task sequence of one role of a CTA pair.
//   Static: t = cid, cid + nclusters, ... (a persistent grid).
//   Dynamic (dynamic task allocation, which "Block Scheduler Code
//   Explained" lists among the scheduler's policies): the grid holds one
//   cluster per task.  A cluster starts with its own task and then takes the
//   tasks of clusters that have not started yet, which the leader's A-load
//   thread cancels one at a time through cluster launch control.  Each
//   response lands in a ring of kClcDepth slots in both CTAs; every other
//   role reads it and frees the slot on the leader, so the claims run at most
//   kClcDepth tasks ahead of the slowest role.  A response that cancelled
//   nothing (or a task past the end) ends every role's sequence at the same
//   point, and no request follows it.
struct PairTasks {
    uint32_t total, step;       // step: nclusters (static) or 0 (dynamic)
    uint4* resp;                // [kClcDepth] responses, this CTA
    uint64_t* full;             // [kClcDepth] response barriers, this CTA
    uint64_t* empty;            // [kClcDepth] slot-free barriers (the leader's are used)
    uint32_t empty_leader;      // cluster address of the leader's empty[0]
    uint32_t peer_full;         // cluster address of the peer's full[0]
    uint32_t i;                 // responses read
    bool pending;               // issuer: a request whose response is unread

    // issuer only: claim the next not-yet-started cluster into slot i
    __device__ __forceinline__ bool request(const WaitCtl& ctl) {
        const uint32_t s = i % kClcDepth, ph = (i / kClcDepth) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, ctl, 9)) return false;
        mbar_arrive_expect_tx(&full[s], 16);
        mbar_arrive_expect_tx_cluster_relaxed(peer_full + s * 8, 16);
        clc_try_cancel_multicast(&resp[s], &full[s]);
        pending = true;
        return true;
    }
    // the task after t (total: none).  role 0: the issuer; 1: a consumer
    // thread; 2: a consumer warp (all lanes call it)
    __device__ __forceinline__ uint32_t next(uint32_t t, bool& ok, uint32_t role, const WaitCtl& ctl) {
        if (step) return t + step;
        const uint32_t s = i % kClcDepth, ph = (i / kClcDepth) & 1u;
        const bool got = role == 2 ? warp_wait(&full[s], ph, ctl, 10) : mbar_wait(&full[s], ph, ctl, 10);
        if (!got) { ok = false; return total; }
        const uint32_t x = clc_cancelled_ctaid_x(&resp[s]);
        const uint32_t nt = x == 0xFFFFFFFFu ? total : min(x >> 1, total);
        ++i;
        if (role == 0) {
            pending = false;
            if (nt < total && !request(ctl)) { ok = false; return total; }
        } else if (role == 1 || (threadIdx.x & 31u) == 0) {
            mbar_arrive_cluster_relaxed(empty_leader + s * 8);
        }
        return nt;
    }
};

// Dequant: one fp32 accumulator (the current K-chunk) in TMEM columns
// [0, BN) and the exact int32 running sums in [BN, 2*BN); otherwise two fp32
// accumulators, so the epilogue of one tile overlaps the MMAs of the next.
template <uint32_t BN, uint32_t STAGES, uint32_t EPI = kEpiStore>
struct PairLayout {
    static constexpr uint32_t EPI_WARPS = pair_epi_warps<EPI>();
    static constexpr uint32_t kACC = EPI == kEpiDequant ? 1 : 2;
    static constexpr uint32_t kABytes = kBM * kLine;            // 128 A rows per CTA
    static constexpr uint32_t kBBytes = (BN / 2) * kLine;       // BN/2 B rows per CTA
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kEpiOff = STAGES * kStageBytes;             // epilogue warps x 4 KB staging
    static constexpr uint32_t kBarOff = kEpiOff + EPI_WARPS * kEpiWarpBytes;
    // full, empty, tfull, tempty, drain, then the task ring's full and empty
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * kACC + 1 + 2 * kClcDepth;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kClcOff = (kMiscOff + 16 + 15) & ~15u;      // kClcDepth x 16-byte responses
    static constexpr uint32_t kTableOff = kClcOff + 16 * kClcDepth;
    static constexpr uint32_t kTmemCols = EPI == kEpiDequant ? 512 : (kACC * BN <= 256 ? 256 : 512);
    static_assert(kACC * BN <= 512 && (EPI == kEpiStore || BN == 256), "TMEM budget");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static constexpr uint32_t smem_bytes(uint32_t groups) { return 1024 + kTableOff + 8 * (groups + 1); }
};

template <uint32_t BN, uint32_t STAGES, uint32_t EPI = kEpiStore>
__global__ void __launch_bounds__(pair_threads<EPI>(), 1) gemm_pair_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = PairLayout<BN, STAGES, EPI>;
    static_assert(EPI == kEpiStore || BN == 256, "dequant: 256-column tiles, 128 columns per epilogue warp");
    constexpr uint32_t ACC = Lay::kACC;
    constexpr uint32_t TM = 2 * kBM;
    constexpr uint32_t BH = BN / 2;                  // B columns held by each CTA
    static_assert(BN == 128 || BN == 256, "BN");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m, &prm.g.ps};
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
    uint64_t* clc_full = drain + 1;
    uint64_t* clc_empty = clc_full + kClcDepth;
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
    // k-blocks of a tile: the group's own count for slice-K (kept in the
    // group table's first G words), else every tile's
    auto tile_kb = [&](uint32_t tag) -> uint32_t { return mode == kModeSliceK ? gt.tile_off[tag] : num_kb; };

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (uint32_t a = 0; a < ACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * pair_epi_warps<EPI>());   // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        for (uint32_t j = 0; j < kClcDepth; ++j) {
            mbar_init(&clc_full[j], 1);
            // every role but the issuer, in both CTAs: A (peer), B (both),
            // MMA, epilogue warps (both)
            mbar_init(&clc_empty[j], 4 + 2 * pair_epi_warps<EPI>());
        }
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
    // set-up above touches no global memory: it overlaps the previous kernel
    griddep_wait();
    griddep_launch_dependents();
    if (mode == kModeGrouped && warp == 2)
        build_group_table(gt, prm.g.group_m, G, N, TM, BN, sa.total_m, err, tiles_smem, lane);
    if (mode == kModeSliceK && warp == 2) {
        // the set-up kernel's per-group k-block counts; bad sizes: no tasks
        const uint32_t bad = prm.g.group_kb[G];
        for (uint32_t g = lane; g < G; g += 32) gt.tile_off[g] = bad ? 0u : prm.g.group_kb[g];
        if (lane == 0 && bad) *tiles_smem = 0;
    }
    __syncwarp();                                    // reconverge lane-0 set-up branches first
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t total_tiles = *tiles_smem;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    if (tl && threadIdx.x == 0) tl[0] = globaltimer_ns();
    const bool dyn = prm.g.dynamic != 0;
    PairTasks tasks{total_tiles, dyn ? 0u : nclusters, reinterpret_cast<uint4*>(smem + Lay::kClcOff), clc_full,
                    clc_empty, map_to_cta(smem_u32(clc_empty), 0), map_to_cta(smem_u32(clc_full), 1), 0, false};

    if (warp == 0 || warp == kPairBWarp) {
        // ------------------------------------------------------ producer --
        // both CTAs: own A half (warp 0) and own B half (warp 6), counted on
        // the leader's full[s]; the leader's A thread is the one arrival
        const uint32_t full_leader = map_to_cta(smem_u32(full), 0);
        constexpr uint32_t tx = Lay::kABytes + Lay::kBBytes;
        const bool is_a = warp == 0;
        uint32_t stage = 0, phase = 0, issued = 0, map_group = 0xFFFFFFFFu;
        bool ok = true;
        const CUtensorMap* map_a = &prm.tmap_a;
        const CUtensorMap* map_b = &prm.tmap_b;
        // single threads issue the loads (cheaper per k-block than a
        // warp-wide loop with one active lane)
        const uint32_t role = (rank == 0 && is_a) ? 0u : 1u;
        if (lane == 0 && dyn && role == 0 && cid < total_tiles) ok = tasks.request(ctl);
        for (uint32_t t = cid; lane == 0 && ok && t < total_tiles; t = tasks.next(t, ok, role, ctl)) {
            const TileInfo ti = tile_info(sa, t, TM, BN, gt);
            const uint32_t a_row = ti.row0 + rank * kBM;
            const uint32_t b_col = ti.n * BN + rank * BH;
            const int32_t zc = static_cast<int32_t>(ti.tag);
            const uint32_t tkb = tile_kb(ti.tag);
            if (mode == kModeSliceK && tkb && ti.tag != map_group) {
                // this group's maps (base at its first K element, K extent
                // its size), written by the set-up kernel
                const uint8_t* gm = prm.g.kmaps + static_cast<uint64_t>(ti.tag) * 256u;
                map_a = reinterpret_cast<const CUtensorMap*>(gm);
                map_b = reinterpret_cast<const CUtensorMap*>(gm + 128);
                tmap_acquire(is_a ? gm : gm + 128);
                map_group = ti.tag;
            }
            // ShuffleK: the K loop of task t starts at k-block t % tkb
            const uint32_t rot = (prm.g.shuffle_k && tkb) ? t % tkb : 0u;
            for (uint32_t kb = 0; kb < tkb; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                {
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    uint8_t* sb_s = sa_s + Lay::kABytes;
                    const uint32_t bar = full_leader + stage * 8;
                    const uint32_t kx = kb + rot;
                    const int32_t k0 = (kx < tkb ? kx : kx - tkb) * bk_elems;
                    if (is_a) {
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                        if (!a_mn) {
                            if (a_rank3) tma_load_3d_pair(sa_s, map_a, bar, k0, a_row, zc);
                            else tma_load_2d_pair(sa_s, map_a, bar, k0, a_row);
                        } else {
                            for (uint32_t j = 0; j < kBM / bk_elems; ++j) {
                                if (a_rank3) tma_load_3d_pair(sa_s + j * bk_elems * kLine, map_a, bar, a_row + j * bk_elems, k0, zc);
                                else tma_load_2d_pair(sa_s + j * bk_elems * kLine, map_a, bar, a_row + j * bk_elems, k0);
                            }
                        }
                    } else if (!b_mn) {
                        if (b_rank3) tma_load_3d_pair(sb_s, map_b, bar, k0, b_col, zc);
                        else tma_load_2d_pair(sb_s, map_b, bar, k0, b_col);
                    } else {
                        for (uint32_t j = 0; j < BH / bk_elems; ++j) {
                            if (b_rank3) tma_load_3d_pair(sb_s + j * bk_elems * kLine, map_b, bar, b_col + j * bk_elems, k0, zc);
                            else tma_load_2d_pair(sb_s + j * bk_elems * kLine, map_b, bar, b_col + j * bk_elems, k0);
                        }
                    }
                    if (tl && is_a && issued < 15) tl[1 + issued] = globaltimer_ns();
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (lane == 0 && tasks.pending) {
            // the issuer gave up with a request in flight: let its response land
            mbar_wait_drain(&clc_full[tasks.i % kClcDepth], (tasks.i / kClcDepth) & 1u, ctl.timeout_ns);
        }
        if (lane == 0 && !ok && rank == 0 && is_a) {
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
            const uint32_t chunk_kb = prm.g.chunk_kb;
            // the whole warp runs the loop (waits are warp-wide); the elected
            // lane (lane 0) issues every MMA and commit
            for (uint32_t t = cid; ok && t < total_tiles; t = tasks.next(t, ok, 2, ctl)) {
              // an empty slice-K group has no MMAs: its epilogue stores zeros
              const uint32_t tkb = mode == kModeSliceK ? tile_kb(tile_info(sa, t, TM, BN, gt).tag) : num_kb;
              const uint32_t nchunks = (tkb + chunk_kb - 1) / chunk_kb;
              // K-chunks (one for plain stores): each fills one accumulator
              for (uint32_t c = 0; ok && c < nchunks; ++c) {
                const uint32_t kb_begin = c * chunk_kb;
                const uint32_t kb_end = min(tkb, kb_begin + chunk_kb);
                if (!warp_wait(&tempty[acc], acc_phase ^ 1u, ctl, 2)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                    if (!warp_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
                        if (tl && mma_kb < 16) tl[16 + mma_kb] = globaltimer_ns();
                        const uint32_t sa_addr = smem_base + stage * Lay::kStageBytes;
                        const uint64_t adesc = smem_desc(sa_addr, a_lbo, 1024, kSwizzle128B);
                        const uint64_t bdesc = smem_desc(sa_addr + Lay::kABytes, b_lbo, 1024, kSwizzle128B);
#pragma unroll
                        for (uint32_t kk = 0; kk < 4; ++kk)
                            umma_f16_pair(d_tmem, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4), idesc,
                                          (kb > kb_begin || kk > 0) ? 1u : 0u);
                        umma_commit_pair_mc(&empty[stage], 0x3);
                    }
                    __syncwarp();
                    ++mma_kb;
                    any_mma = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (elect_one()) umma_commit_pair_mc(&tfull[acc], 0x3);
                __syncwarp();
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
              }
            }
            if (lane == 0 && !ok && any_mma) {
                // every tcgen05 op issued so far must finish before TMEM is freed
                umma_commit_pair_mc(drain, 0x1);
                mbar_wait_drain(drain, 0, ctl.timeout_ns);
            }
        }
    } else if ((warp >= 2 && warp < 6) || (EPI == kEpiDequant && warp >= 7 && warp < 11)) {
        // ---------------------------------------------- epilogue (both) --
        const bool hi = warp >= 7;                       // dequant: the upper 128 columns
        if (!hi) prefetch_operands(prm.g, threadIdx.x - 64, 128);
        constexpr uint32_t kCols = EPI == kEpiDequant ? BN / 2 : BN;   // columns this warp finishes
        const uint32_t col_off = hi ? BN / 2 : 0u;
        const uint32_t q = warp & 3u;                    // TMEM lane quarter of this warp
        const uint32_t wrow = rank * kBM + q * 32;       // first row of this warp in the 256-row tile
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec, acc_vec = prm.g.acc_vec;
        uint8_t* const epi_stage = smem + Lay::kEpiOff + (hi ? 4u + q : q) * kEpiWarpBytes;
        uint8_t* const C = prm.g.C;
        const int64_t ldc = prm.g.ldc, c_bs = prm.g.c_batch_stride;
        const float* scale_a = prm.g.scale_a;
        const float* scale_b = prm.g.scale_b;
        int32_t* const acc_out = prm.g.acc_out;
        uint32_t* const trace = prm.g.trace;
        const uint32_t trace_cap = prm.g.trace_cap;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        const uint32_t tempty_leader = map_to_cta(smem_u32(tempty), 0);
        const uint32_t chunk_kb = prm.g.chunk_kb;
        uint32_t acc = 0, acc_phase = 0, ep_tile = 0;
        bool ok = true;
        for (uint32_t t = cid; ok && t < total_tiles; t = tasks.next(t, ok, 2, ctl)) {
            const TileInfo ti = tile_info(sa, t, TM, BN, gt);
            if (trace && rank == 0 && warp == 2 && lane == 0) {
                if (t < trace_cap) {
                    uint32_t* tr = trace + static_cast<uint64_t>(t) * 5;
                    tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
                } else {
                    atomicOr(&err[0], kErrTraceOverflow);
                }
            }
            const uint32_t rows_valid = ti.m_act > wrow ? min(32u, ti.m_act - wrow) : 0u;   // warp-uniform
            const int64_t cbase = (mode == kModeBatched || mode == kModeSliceK) ? static_cast<int64_t>(ti.tag) * c_bs : 0;
            uint8_t* const cwarp = C + (cbase + static_cast<int64_t>(ti.row0 + wrow) * ldc) * csize;
            const uint32_t n0 = ti.n * BN + col_off;     // first output column of this warp
            const uint32_t n_act = ti.n_act > col_off ? ti.n_act - col_off : 0u;
            // dequant: exact int32 running sums of this warp's rows and columns
            const uint32_t run_t = tmem_base + ((q * 32) << 16) + BN + col_off;
            const uint32_t nchunks = (tile_kb(ti.tag) + chunk_kb - 1) / chunk_kb;
            if (nchunks == 0) {
                // an empty slice-K group: C_g (and its accumulators) are zero
                uint32_t z[32];
#pragma unroll
                for (uint32_t j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll 1
                for (uint32_t cc = 0; rows_valid && cc < kCols / 32 && cc * 32 < n_act; ++cc) {
                    store_chunk_coalesced(epi_stage, c_type, c_vec, cwarp + static_cast<int64_t>(n0 + cc * 32) * csize,
                                          ldc * csize, rows_valid, min(32u, n_act - cc * 32), z, lane);
                    if (EPI == kEpiDequant && acc_out) {
                        uint8_t* awarp = reinterpret_cast<uint8_t*>(
                            acc_out + cbase + static_cast<int64_t>(ti.row0 + wrow) * ldc + n0 + cc * 32);
                        store_chunk_coalesced(epi_stage, kOutS32, acc_vec, awarp, ldc * 4, rows_valid,
                                              min(32u, n_act - cc * 32), z, lane);
                    }
                }
                continue;
            }
            for (uint32_t c = 0; c < nchunks; ++c) {
                if (!warp_wait(&tfull[acc], acc_phase, ctl, 4)) { ok = false; break; }
                tc_fence_after();
                if (tl && warp == 2 && lane == 0 && c == 0 && ep_tile < 8) tl[32 + ep_tile] = globaltimer_ns();
                const uint32_t taddr = tmem_base + ((q * 32) << 16) + acc * BN + col_off;
                if (EPI == kEpiStore) {
#pragma unroll 1
                    for (uint32_t cc = 0; cc < kCols / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + cc * 32, v);
                        if (rows_valid && cc * 32 < n_act)
                            store_chunk_coalesced(epi_stage, c_type, c_vec,
                                                  cwarp + static_cast<int64_t>(n0 + cc * 32) * csize, ldc * csize,
                                                  rows_valid, min(32u, n_act - cc * 32), v, lane);
                    }
                } else {
                    // fold the chunk (an exact integer in fp32) into the running
                    // sums.  The accumulator is released as soon as the chunk is
                    // in registers, so the next chunk's MMAs overlap the update
                    // of the running sums (other TMEM columns).
                    int32_t ci[EPI == kEpiDequant ? kCols : 1];
#pragma unroll
                    for (uint32_t cc = 0; cc < kCols / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + cc * 32, v);
#pragma unroll
                        for (uint32_t j = 0; j < 32; ++j)
                            ci[(EPI == kEpiDequant ? cc * 32 + j : 0)] = __float2int_rn(__uint_as_float(v[j]));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
#pragma unroll
                    for (uint32_t cc = 0; cc < kCols / 32; ++cc) {
                        uint32_t r[32];
                        if (c > 0) tmem_ld_32x32b_x32(run_t + cc * 32, r);
#pragma unroll
                        for (uint32_t j = 0; j < 32; ++j)
                            r[j] = static_cast<uint32_t>((c > 0 ? static_cast<int32_t>(r[j]) : 0) +
                                                         ci[(EPI == kEpiDequant ? cc * 32 + j : 0)]);
                        tmem_st_32x32b_x32(run_t + cc * 32, r);
                    }
                }
                if (EPI == kEpiStore) {
                    // the accumulator's reads are complete (tcgen05.wait::ld):
                    // a relaxed arrival releases it, with no data to publish
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
                }
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;
            if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[40 + ep_tile] = globaltimer_ns();
            ++ep_tile;
            if (EPI == kEpiDequant && rows_valid) {
                // acc * scale_a[row] * scale_b[col] in fp32, rounded once to bf16
                tc_fence_after();
                const uint32_t grow = ti.row0 + wrow + lane;
                // slice-K: this group's row scales (sa_group_stride 0 otherwise)
                const float sa_row =
                    lane < rows_valid ? scale_a[static_cast<int64_t>(ti.tag) * prm.g.sa_group_stride + grow] : 0.f;
                // grouped: this group's column scales (tag = group; 0 for plain problems)
                const float* sb_row = scale_b + static_cast<int64_t>(ti.tag) * prm.g.sb_group_stride;
#pragma unroll 1
                for (uint32_t cc = 0; cc < kCols / 32; ++cc) {
                    if (cc * 32 >= n_act) break;
                    const uint32_t col0 = n0 + cc * 32;
                    const uint32_t nv = min(32u, n_act - cc * 32);
                    uint32_t r[32], v[32];
                    tmem_ld_32x32b_x32(run_t + cc * 32, r);
#pragma unroll
                    for (uint32_t j = 0; j < 32; ++j) {
                        const float sb = j < nv ? __ldg(sb_row + col0 + j) : 0.f;
                        v[j] = __float_as_uint(static_cast<float>(static_cast<int32_t>(r[j])) * sa_row * sb);
                    }
                    store_chunk_coalesced(epi_stage, c_type, c_vec, cwarp + static_cast<int64_t>(col0) * csize,
                                          ldc * csize, rows_valid, nv, v, lane);
                    if (acc_out) {
                        uint8_t* awarp = reinterpret_cast<uint8_t*>(acc_out + cbase + static_cast<int64_t>(ti.row0 + wrow) * ldc + col0);
                        store_chunk_coalesced(epi_stage, kOutS32, acc_vec, awarp, ldc * 4, rows_valid, nv, r, lane);
                    }
                }
            }
        }
    }

    if (tl && lane == 0 && warp <= 2) tl[48 + warp] = globaltimer_ns();
    // single-lane roles leave their warps diverged: reconverge every warp
    // first, so that the barrier counts each warp once; the cluster barrier
    // also orders this CTA's own warps before TMEM is freed
    __syncwarp();
    tc_fence_before();
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
// [p*kb/S, (p+1)*kb/S) of it exactly as gemm_pair_kernel does, into one TMEM
// accumulator of 128 rows per CTA.
//
// The S fp32 partial tiles are summed on chip.  Split g finishes columns
// [g*W, (g+1)*W) (W = BN/S) of each CTA's 128 rows.  Once its pair's MMAs are
// done (the stage ring is then idle), every epilogue warp copies, for each
// other split g, its 32 rows of its share of g's columns into the ring, and
// one bulk copy moves them into a receive slot of the CTA of split g (same
// half), completing on that CTA's receive barrier of the same warp.  The
// receive slots sit outside the ring, so a sender never waits for the
// receiver.  The warp then adds the S-1 slots it received to its own rows of
// its share of its own columns, rounds once and stores them through the
// coalesced epilogue.  The epilogue warps are 2-5 and, when the ring has room
// (W >= 64), also 0, 1, 6 and 7 once their loads and MMAs are issued: two
// warps per TMEM lane quarter, each with half of the columns.  All send and
// finish in parallel; nothing goes through global memory and no second
// kernel runs.
//
// Shared-memory rows of a partial (W fp32) keep their 16-byte granules
// XOR-swizzled by row (granule c at c ^ (row % 8)), so both the row-per-lane
// writes and the row-per-lane reads are conflict-free.
template <uint32_t BN, uint32_t STAGES, uint32_t S>
struct SplitLayout {
    static constexpr uint32_t kABytes = kBM * kLine;
    static constexpr uint32_t kBBytes = (BN / 2) * kLine;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kW = BN / S;                         // columns each split finishes
    static constexpr uint32_t kSlotBytes = 32 * kW * 4;            // 32 rows of W columns
    static constexpr uint32_t kSlots = 4 * (S - 1);                // per CTA, sent and received
    static constexpr uint32_t kRecvOff = STAGES * kStageBytes;
    static constexpr uint32_t kRecvBytes = kSlots * kSlotBytes;
    // Epilogue groups: warps 2-5, and (kEH = 2) warps 0, 1, 6, 7 once their
    // loads and MMAs are issued; the group of warp w finishes columns
    // [h*kWH, (h+1)*kWH) of each split's W in TMEM lane quarter w % 4.  The
    // second group stages its stores in the idle ring, after the send staging.
    static constexpr uint32_t kEH =
        (kW >= 64 && kSlots * kSlotBytes + 4 * kEpiWarpBytes <= STAGES * kStageBytes) ? 2u : 1u;
    static constexpr uint32_t kWH = kW / kEH;
    static constexpr uint32_t kSubBytes = 32 * kWH * 4;            // one warp's rows of its kWH columns
    static constexpr uint32_t kEpi1Off = kSlots * kSlotBytes;      // second group's store staging (ring)
    static constexpr uint32_t kThreads = kEH == 2 ? 256u : 224u;
    static constexpr uint32_t kEpiOff = kRecvOff + kRecvBytes;
    static constexpr uint32_t kBarOff = kEpiOff + 4 * kEpiWarpBytes;
    // full, empty, tfull, drain, recv[4 * kEH]
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 + 4 * kEH;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kTmemCols = BN;
    static constexpr uint32_t smem_bytes() { return 1024 + kMiscOff + 16; }
    static_assert(S == 2 || S == 4, "splits");
    static_assert(kW % 32 == 0 && kWH % 32 == 0, "whole 32-column chunks per split and group");
    static_assert(kSlots * kSlotBytes <= STAGES * kStageBytes, "sender staging reuses the ring");
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(smem_bytes() <= 232448, "shared memory per CTA");
};

template <uint32_t BN, uint32_t STAGES, uint32_t S>
__global__ void __launch_bounds__(256, 1) gemm_pair_splitk_kernel(const __grid_constant__ GemmParams prm) {
    using SL = SplitLayout<BN, STAGES, S>;
    constexpr uint32_t TM = 2 * kBM;
    constexpr uint32_t BH = BN / 2;
    static_assert(BN == 128 || BN == 256, "BN");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m, &prm.g.ps};
    const uint32_t num_kb = prm.g.num_kb;
    const uint32_t a_mn = prm.g.a.mn_major, b_mn = prm.g.b.mn_major;
    uint32_t* const err = prm.g.err;
    constexpr uint32_t bk_elems = 64;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* drain = bars + 2 * STAGES + 1;
    uint64_t* recv = bars + 2 * STAGES + 2;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + SL::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    uint64_t* const tl = prm.g.timeline ? prm.g.timeline + static_cast<uint64_t>(blockIdx.x) * 64 : nullptr;
    const uint64_t t_entry = globaltimer_ns();
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
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        for (uint32_t o = 0; o < 4 * SL::kEH; ++o) mbar_init(&recv[o], 1);
        *abort_flag = 0;
        fence_barrier_init();
        // the receive barrier of each epilogue warp expects the S-1 partials of its rows
        for (uint32_t o = 0; o < 4 * SL::kEH; ++o) mbar_arrive_expect_tx(&recv[o], (S - 1) * SL::kSubBytes);
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&prm.tmap_a);
        prefetch_tmap(&prm.tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, SL::kTmemCols);
        tmem_relinquish_pair();
    }
    __syncwarp();                                    // reconverge lane-0 set-up branches first
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                  // barriers of every CTA initialised
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    GroupTable gt{nullptr, nullptr, 0};
    TileInfo ti{};
    if (has_tile) ti = tile_info(sa, t, TM, BN, gt);
    if (has_tile && has_k && warp >= 2 && warp < 6) {
        // the epilogue warps (idle until the accumulator is ready) pull this
        // CTA's first k-blocks into L2 while the previous kernel finishes
        const uint32_t nk = min(4u, kb_end - kb_begin);
        prefetch_tile_l2(prm.g.a, ti.row0 + half * kBM, kBM, prm.g.M, kb_begin, nk, prm.g.K, threadIdx.x - 64, 128);
        prefetch_tile_l2(prm.g.b, ti.n * BN + half * BH, BH, prm.g.N, kb_begin, nk, prm.g.K, threadIdx.x - 64, 128);
    }
    // set-up above (the tile's coordinates come from the arguments alone,
    // and an L2 prefetch reads nothing into the SM) overlaps the previous
    // kernel
    griddep_wait();
    if (tl && threadIdx.x == 0) tl[44] = globaltimer_ns();
    griddep_launch_dependents();
    if (tl && threadIdx.x == 0) { tl[0] = t_entry; tl[1] = globaltimer_ns(); }

    if ((warp == 0 || warp == kPairBWarp) && lane == 0 && has_tile) {
        // ------------------------------------------------------ producer --
        // A half by warp 0 (the pair leader's is the one arrival), B half by warp 6
        const bool is_a = warp == 0;
        const uint32_t full_leader = map_to_cta(smem_u32(full), leader);
        constexpr uint32_t tx = SL::kABytes + SL::kBBytes;
        const uint32_t a_row = ti.row0 + half * kBM;
        const uint32_t b_col = ti.n * BN + half * BH;
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        // ShuffleK: this split's range starts at (task + split) % its k-blocks
        const uint32_t nk = kb_end - kb_begin;
        const uint32_t rot = (prm.g.shuffle_k && nk) ? (t + split) % nk : 0u;
        for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
            // the ring starts empty: only a stage being reused is waited for
            if (issued >= STAGES && !mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
            uint8_t* sa_s = smem + stage * SL::kStageBytes;
            uint8_t* sb_s = sa_s + SL::kABytes;
            const uint32_t bar = full_leader + stage * 8;
            const uint32_t kx = kb + rot;
            const int32_t k0 = (kx < kb_end ? kx : kx - nk) * bk_elems;
            if (is_a) {
                if (half == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                if (!a_mn) tma_load_2d_pair(sa_s, &prm.tmap_a, bar, k0, a_row);
                else
                    for (uint32_t j = 0; j < kBM / bk_elems; ++j)
                        tma_load_2d_pair(sa_s + j * bk_elems * kLine, &prm.tmap_a, bar, a_row + j * bk_elems, k0);
            } else if (!b_mn) {
                tma_load_2d_pair(sb_s, &prm.tmap_b, bar, k0, b_col);
            } else {
                for (uint32_t j = 0; j < BH / bk_elems; ++j)
                    tma_load_2d_pair(sb_s + j * bk_elems * kLine, &prm.tmap_b, bar, b_col + j * bk_elems, k0);
            }
            if (tl && is_a && issued < 14) tl[2 + issued] = globaltimer_ns();
            ++issued;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok && half == 0 && is_a) {
            uint32_t s = stage, ph = phase;
            const uint32_t pending = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < pending; ++i) {
                if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
            }
        }
    } else if (warp == 1 && has_tile && has_k && half == 0) {
        // ------------------------------------- MMA issuer (pair leaders) --
        // the whole warp runs the loop; the elected lane (lane 0) issues
        const uint32_t a_lbo = a_mn ? bk_elems * kLine : 16u;
        const uint32_t b_lbo = b_mn ? bk_elems * kLine : 16u;
        const uint32_t a_step = a_mn ? 16u * kLine : 32u;
        const uint32_t b_step = b_mn ? 16u * kLine : 32u;
        const uint32_t idesc = idesc_f16(prm.g.ab_fmt, a_mn, b_mn, TM, BN);
        const uint32_t smem_base = smem_u32(smem);
        uint32_t stage = 0, phase = 0;
        bool ok = true, any_mma = false;
        for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
            if (!warp_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
                const uint32_t sa_addr = smem_base + stage * SL::kStageBytes;
                const uint64_t adesc = smem_desc(sa_addr, a_lbo, 1024, kSwizzle128B);
                const uint64_t bdesc = smem_desc(sa_addr + SL::kABytes, b_lbo, 1024, kSwizzle128B);
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    umma_f16_pair(tmem_base, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4), idesc,
                                  (kb > kb_begin || kk > 0) ? 1u : 0u);
                umma_commit_pair_mc(&empty[stage], pair_mask);
                if (tl && kb - kb_begin < 16) tl[16 + kb - kb_begin] = globaltimer_ns();
            }
            __syncwarp();
            any_mma = true;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (lane == 0) {                                 // the lane that issued the MMAs
            if (ok) umma_commit_pair_mc(tfull, pair_mask);
            else if (any_mma) {
                umma_commit_pair_mc(drain, static_cast<uint16_t>(1u << crank));
                mbar_wait_drain(drain, 0, ctl.timeout_ns);
            }
        }
    }
    __syncwarp();                                        // reconverge the single-lane load warps
    const bool epi_main = warp >= 2 && warp < 6;
    if ((epi_main || (SL::kEH == 2 && (warp < 2 || warp >= 6))) && has_tile) {
        // ----------------------------------------------------- epilogue --
        const uint32_t q = warp & 3u;                    // TMEM lane quarter of this warp
        const uint32_t h = epi_main ? 0u : 1u;           // column group of this warp
        const uint32_t taddr = tmem_base + ((q * 32) << 16);
        constexpr uint32_t W = SL::kW, WH = SL::kWH;
        const uint32_t qh = q * SL::kEH + h;             // receive barrier and slot group
        // this warp's rows are final once its pair's MMAs are done
        bool acc_ok = true;
        if (has_k) acc_ok = warp_wait(tfull, 0, ctl, 4);
        tc_fence_after();
        if (tl && warp == 2 && lane == 0) tl[32] = globaltimer_ns();
        const bool own_valid = acc_ok && has_k;          // else this split's partial counts as zero
        // send: for every other split g, this warp's rows of its group of g's columns
        uint32_t gi = 0;
#pragma unroll 1
        for (uint32_t g = 0; g < S; ++g) {
            if (g == split) continue;
            uint8_t* stage_rows = smem + (qh * (S - 1) + gi) * SL::kSubBytes;
            uint8_t* my_row = stage_rows + lane * (WH * 4);
#pragma unroll 1
            for (uint32_t cc = 0; cc < WH / 32; ++cc) {
                uint32_t v[32];
                if (own_valid) tmem_ld_32x32b_x32(taddr + g * W + h * WH + cc * 32, v);
                else {
#pragma unroll
                    for (uint32_t j = 0; j < 32; ++j) v[j] = 0u;
                }
#pragma unroll
                for (uint32_t gg = 0; gg < 8; ++gg) {
                    const uint32_t granule = (cc * 8 + gg) ^ (lane & 7u);
                    *reinterpret_cast<uint4*>(my_row + granule * 16) =
                        make_uint4(v[4 * gg], v[4 * gg + 1], v[4 * gg + 2], v[4 * gg + 3]);
                }
            }
            fence_proxy_async_smem();                    // generic writes -> the bulk copy's reads
            __syncwarp();
            if (lane == 0) {
                const uint32_t dest = 2 * g + half;      // split g, same half
                const uint32_t slot = qh * (S - 1) + (split < g ? split : split - 1);
                const uint32_t dst = map_to_cta(smem_u32(smem + SL::kRecvOff + slot * SL::kSubBytes), dest);
                const uint32_t bar = map_to_cta(smem_u32(&recv[qh]), dest);
                bulk_copy_to_cluster(dst, stage_rows, SL::kSubBytes, bar);
                bulk_commit_group();
            }
            ++gi;
        }
        if (tl && warp == 2 && lane == 0) tl[34] = globaltimer_ns();
        // finish: own rows of own columns plus the S-1 received partials
        const bool got = warp_wait(&recv[qh], 0, ctl, 5);
        if (tl && warp == 2 && lane == 0) tl[33] = globaltimer_ns();
        if (tl && lane == 0 && h == 0) tl[48 + q] = globaltimer_ns();
        const uint8_t* slots = smem + SL::kRecvOff + qh * (S - 1) * SL::kSubBytes + lane * (WH * 4);
        const uint32_t wrow = half * kBM + q * 32;       // first row of this warp in the tile
        const uint32_t rows_valid = ti.m_act > wrow ? min(32u, ti.m_act - wrow) : 0u;
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        const int64_t ldc = prm.g.ldc;
        uint8_t* const cwarp = prm.g.C + static_cast<int64_t>(ti.row0 + wrow) * ldc * csize;
        uint8_t* const epi_stage = smem + (h ? SL::kEpi1Off : SL::kEpiOff) + q * kEpiWarpBytes;
#pragma unroll 1
        for (uint32_t cc = 0; cc < WH / 32; ++cc) {
            uint32_t v[32];
            if (own_valid) tmem_ld_32x32b_x32(taddr + split * W + h * WH + cc * 32, v);
            else {
#pragma unroll
                for (uint32_t j = 0; j < 32; ++j) v[j] = 0u;
            }
            if (got) {
#pragma unroll
                for (uint32_t si = 0; si < S - 1; ++si) {
#pragma unroll
                    for (uint32_t gg = 0; gg < 8; ++gg) {
                        const uint32_t granule = (cc * 8 + gg) ^ (lane & 7u);
                        const uint4 x = *reinterpret_cast<const uint4*>(slots + si * SL::kSubBytes + granule * 16);
                        v[4 * gg] = __float_as_uint(__uint_as_float(v[4 * gg]) + __uint_as_float(x.x));
                        v[4 * gg + 1] = __float_as_uint(__uint_as_float(v[4 * gg + 1]) + __uint_as_float(x.y));
                        v[4 * gg + 2] = __float_as_uint(__uint_as_float(v[4 * gg + 2]) + __uint_as_float(x.z));
                        v[4 * gg + 3] = __float_as_uint(__uint_as_float(v[4 * gg + 3]) + __uint_as_float(x.w));
                    }
                }
            }
            const uint32_t col = split * W + h * WH + cc * 32;   // column within the tile
            if (rows_valid && col < ti.n_act)
                store_chunk_coalesced(epi_stage, c_type, c_vec, cwarp + static_cast<int64_t>(ti.n * BN + col) * csize,
                                      ldc * csize, rows_valid, min(32u, ti.n_act - col), v, lane);
        }
        if (tl && lane == 0 && h == 0) tl[40 + q] = globaltimer_ns();
        if (lane == 0) bulk_wait_read_all();             // the ring may not be left while being read
        if (prm.g.trace && split == 0 && half == 0 && q == 0 && h == 0 && lane == 0 && t < prm.g.trace_cap) {
            uint32_t* tr = prm.g.trace + static_cast<uint64_t>(t) * 5;
            tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
        }
    }

    if (tl && threadIdx.x == 64) tl[36] = globaltimer_ns();
    // single-lane roles leave their warps diverged: reconverge every warp
    // first, so that the barrier counts each warp once.  The cluster barrier
    // also orders this CTA's own warps (a block barrier before it only adds
    // latency): no CTA leaves, and no TMEM is freed, while any thread of the
    // cluster may still touch it.  Its arrival is relaxed: every access a CTA
    // makes to another's shared memory has completed before it gets here (the
    // partials it sent were counted on the receivers' barriers, which they
    // waited for, and its bulk copies have finished reading its own ring), so
    // there is nothing to release, and a release arrival would first wait for
    // this CTA's global stores of C to drain.
    __syncwarp();
    tc_fence_before();
    cluster_sync_relaxed_arrive();
    if (tl && threadIdx.x == 0) tl[39] = globaltimer_ns();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, SL::kTmemCols);
    }
    if (tl && threadIdx.x == 0) tl[37] = globaltimer_ns();
}

}  // namespace bst
