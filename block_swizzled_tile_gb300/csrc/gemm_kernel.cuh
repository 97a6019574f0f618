// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks the task indices t = blockIdx.x, blockIdx.x + grid,
// ... ; each task index is turned into an output tile by the block-swizzle
// scheduler (sched.cuh, "Block Scheduler Code Explained" sections 4-7).
// Roles inside the CTA (224 threads, 256 for MXFP8):
//   warp 0     producer: per k-block waits for a free shared-memory stage and
//              fills it (lane 0 issues the A loads by TMA; the warp copies
//              operands TMA cannot take by cp.async) -- the counterpart of the
//              GM->L1 copies of "Block Dispatch Policies" (MmadAtlasA2Preload
//              / PreloadAsync: the producer runs ahead across tile and group
//              boundaries, i.e. inter-block and inter-group preloading).
//              Lane 0 of warp 6 (7 for MXFP8) issues the B loads; for MXFP8,
//              warp 6 lays out the scale factors.  When an fp16/bf16 operand
//              cannot be fetched by TMA, warp 6 instead shares the cp.async
//              copies with warp 0 (each takes every other group of lines): a
//              warp issues such copies about one per 70 ns, so two warps cut
//              a misaligned tile's load time by a third.
//   warp 1     MMA issuer: the whole warp waits on each stage, lane 0 issues
//              tcgen05.mma into a TMEM accumulator and releases the stage with
//              tcgen05.commit.
//   warps 2-5  epilogue: TMEM -> registers -> global, with the tail tile cut
//              by GetActualBlockShape (section 4.6); the accumulator is
//              double-buffered so the epilogue of tile i overlaps the MMAs of
//              tile i+1 (the uintflag / L0C overlap of MmadAtlasA2Pingpong).
//
// Shared-memory stage layout (STAGES copies): A tile 128 rows x 128 bytes,
// then B tile BN rows x 128 bytes, both in the 128-byte-swizzled layout TMA
// writes.  A "line" is 128 bytes: for K-contiguous operands one row of the
// matrix over one k-block (64 x 16-bit or 128 x 8-bit elements); for
// MN-contiguous operands one k of a 64/128-element MN atom.
//
// All kernel arguments are read into registers once at entry; the loops then
// touch no parameter memory (the inline PTX that orders shared memory would
// otherwise force every field to be re-read after each such statement).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"
#include "sched.cuh"

namespace bst {

enum : uint32_t { kKindF16 = 0, kKindMXF8 = 1 };
enum : uint32_t { kEpiStore = 0, kEpiDequant = 1 };
// kModeSliceK: groups along K ("Block Dispatch Policies",
// 05_grouped_matmul_slice_k); group g is batch g of the scheduler, with its
// own tensor maps (kmaps) and k-block count (group_kb).
enum : uint32_t { kModePlain = 0, kModeBatched = 1, kModeGrouped = 2, kModeSliceK = 3 };
enum : uint32_t { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2, kOutS32 = 3 };   // kOutS32: raw int32 (device side only)

constexpr uint32_t kBM = 128;          // tile rows = TMEM lanes
constexpr uint32_t kLine = 128;        // bytes per k-block line
constexpr uint32_t kNumThreads = 192;   // CTA-pair kernels: warps 0 TMA, 1 MMA, 2-5 epilogue
constexpr uint32_t kScaleWarp = 6;      // MXFP8 only: a 7th warp copies scale factors
// One-CTA kernels add a warp whose lane 0 issues the B loads: one thread
// issues about one TMA (or one mbarrier arrive) per 0.1-0.15 us, so a single
// issuing thread cannot feed a 128 x 128 tile's MMAs (one k-block per
// 0.14 us); two threads on two warps issue in parallel.
template <uint32_t KIND>
constexpr uint32_t b_warp_for() { return KIND == 1 ? 7u : 6u; }
template <uint32_t KIND>
constexpr uint32_t threads_for() { return (b_warp_for<KIND>() + 1) * 32; }
// Shared-memory staging of one epilogue warp: a 32 x 32 chunk of 4-byte values.
constexpr uint32_t kEpiWarpBytes = 32 * 32 * 4;
constexpr uint32_t kMaxGroups = 1024;

struct OperandDesc {
    const uint8_t* ptr;
    int64_t ld;            // elements
    int64_t batch_stride;  // elements
    uint32_t mn_major;     // 1: the M (or N) index is contiguous
    uint32_t use_tma;
    uint32_t vec_bytes;    // cp.async / plain-load vector width when !use_tma
    uint32_t tma_rank;     // 2, or 3 when the tensor map has a batch/group dimension
    uint32_t rows2;        // MN-major B with a pitch 8 bytes off a multiple of 16: loaded by TMA
                           // through the two-row view (tmap_sfa: even rows, tmap_sfb: odd rows)
};

// Every scalar argument of the kernel.
struct GemmArgs {
    OperandDesc a, b;
    uint32_t M, N, K;
    uint32_t batch;
    uint32_t mode;
    uint32_t ab_fmt;        // kind::f16 operand format: 0 f16, 1 bf16
    uint32_t esize;         // operand element bytes: 2 or 1
    uint32_t swz_offset, swz_dir;
    uint32_t num_kb;        // k-blocks per tile
    uint32_t chunk_kb;      // k-blocks per accumulation chunk
    uint32_t total_tiles;   // plain / batched (grouped: computed in the kernel)
    const int32_t* group_m;
    uint32_t G;
    uint32_t total_m;
    uint8_t* C;
    int64_t ldc;
    int64_t c_batch_stride;
    uint32_t c_type;
    PlainSched ps;          // plain / batched: the scheduler for the launched tile shape
    uint32_t c_vec;         // widest store (16, 8, 4 or 2 bytes) C's base, pitch and batch stride allow
    uint32_t acc_vec;       // the same for acc_out (int32 accumulators)
    const float* scale_a;
    const float* scale_b;
    int64_t sb_group_stride;   // grouped dequant: elements between the groups' scale_b rows
    int64_t sa_group_stride;   // slice-K dequant: elements between the groups' scale_a rows
    const uint8_t* kmaps;      // slice-K: per group 256 bytes, the A then the B tensor map
    const uint32_t* group_kb;  // slice-K: k-blocks of each group, then a status word (non-zero: bad sizes)
    uint32_t dynamic;          // CTA-pair kernels: tasks claimed through cluster launch control
    uint32_t shuffle_k;        // each tile starts its K loop at k-block (task % k-blocks)
    int32_t* acc_out;
    const uint8_t* sfa;
    const uint8_t* sfb;
    uint32_t sf_ld;         // bytes per row of sfa / sfb (K / 32)
    uint32_t sf_tma;        // 1: scale factors arrive by TMA (tmap_sfa / tmap_sfb), 16 bytes per row per 4 k-blocks
    uint32_t* trace;
    uint32_t trace_cap;     // tasks the trace buffer holds
    uint64_t* timeline;     // optional: 64 %globaltimer stamps per CTA
    uint32_t* err;
    uint64_t timeout_ns;
    // operand byte ranges pulled into L2 at kernel start (small problems,
    // whose loads would otherwise each wait for DRAM); bytes 0 = none
    const uint8_t* pf_ptr[4];
    uint64_t pf_bytes[4];
};

// Each CTA's epilogue threads (idle until the first accumulator is ready)
// issue L2 prefetches for an interleaved 1/grid share of the ranges, so every
// line is requested once and the DRAM fetch of the whole footprint starts
// immediately instead of trickling in behind the TMA loads.
__device__ __forceinline__ void prefetch_operands(const GemmArgs& g, uint32_t tid, uint32_t nthreads) {
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * nthreads;
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        const uint64_t lines = (g.pf_bytes[r] + 127) / 128;
        for (uint64_t L = static_cast<uint64_t>(blockIdx.x) * nthreads + tid; L < lines; L += stride)
            prefetch_l2(g.pf_ptr[r] + L * 128);
    }
}

// L2 prefetch of the first k-blocks of one operand tile: `rows` rows of the
// tile starting at mn0 (below mn_lim), k-blocks [kb0, kb0 + nkb) (of 64
// 16-bit elements, below K), one 128-byte line each, spread over `nthreads`
// threads.  Every prefetched address is an element that exists.  A
// prefetch reads nothing into the SM and L2 stays coherent with whatever an
// earlier kernel still writes, so this may run before griddepcontrol.wait:
// it only moves the DRAM latency of the first loads off the critical path.
__device__ __forceinline__ void prefetch_tile_l2(const OperandDesc& od, uint32_t mn0, uint32_t rows, uint32_t mn_lim,
                                                 uint32_t kb0, uint32_t nkb, uint32_t K, uint32_t tid,
                                                 uint32_t nthreads) {
    if (od.mn_major) {
        // line = one k of a 64-element MN atom
        const uint32_t atoms = rows / 64;
        for (uint32_t L = tid; L < atoms * nkb * 64; L += nthreads) {
            const uint32_t k = kb0 * 64 + L % (nkb * 64), mn = mn0 + (L / (nkb * 64)) * 64;
            if (k < K && mn < mn_lim) prefetch_l2(od.ptr + (static_cast<int64_t>(k) * od.ld + mn) * 2);
        }
    } else {
        // line = one MN row over one k-block
        for (uint32_t L = tid; L < rows * nkb; L += nthreads) {
            const uint32_t k = (kb0 + L % nkb) * 64, mn = mn0 + L / nkb;
            if (k < K && mn < mn_lim) prefetch_l2(od.ptr + (static_cast<int64_t>(mn) * od.ld + k) * 2);
        }
    }
}

struct GemmParams {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;
    CUtensorMap tmap_sfa;   // MXFP8 scale factors as uint8 [rows, K/32], boxes of 16 bytes x 128 / BN rows;
                            // fp16/bf16 with b.rows2: B's even rows (boxes of 64 x 32)
    CUtensorMap tmap_sfb;   // ... fp16/bf16 with b.rows2: B's odd rows (boxes of 72 x 32, 8 bytes early)
    GemmArgs g;
};

template <uint32_t BN, uint32_t STAGES, uint32_t ACC, uint32_t KIND, uint32_t SPLIT = 1>
struct GemmLayout {
    static constexpr uint32_t kABytes = kBM * kLine;
    static constexpr uint32_t kBBytes = BN * kLine;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kSfaBytes = KIND == kKindMXF8 ? 512u : 0u;
    static constexpr uint32_t kSfbBytes = KIND == kKindMXF8 ? BN * 4u : 0u;
    static constexpr uint32_t kSfStageBytes = kSfaBytes + kSfbBytes;
    static constexpr uint32_t kSfOff = STAGES * kStageBytes;
    // MXFP8: two raw scale slots, each 16 bytes (4 k-blocks of E8M0 codes) of
    // the tile's 128 A rows and BN B rows, as TMA delivers them
    static constexpr uint32_t kRawRowsA = 128;
    static constexpr uint32_t kRawSlotBytes = KIND == kKindMXF8 ? (kRawRowsA + BN) * 16u : 0u;
    static constexpr uint32_t kRawOff = (kSfOff + STAGES * kSfStageBytes + 1023) & ~1023u;
    // 4 epilogue warps x 4 KB staging; split-K stages its stores in the idle
    // ring instead (after the main loop), which leaves room for a deeper ring
    static constexpr uint32_t kEpiOff = kRawOff + 2 * kRawSlotBytes;
    static constexpr uint32_t kBarOff = kEpiOff + (SPLIT > 1 ? 0u : 4 * kEpiWarpBytes);
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * ACC + 1 + 4 + 8; // ..., drain, raw_full[4], recv[8]
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kTableOff = (kMiscOff + 16 + 15) & ~15u;
    // TMEM: ACC accumulators of BN fp32 columns, then (MXFP8) per stage 4
    // columns of A scale factors and BN/32 of B scale factors
    static constexpr uint32_t kSfCols = KIND == kKindMXF8 ? (4 + BN / 32) : 0;
    static constexpr uint32_t kColsUsed = ACC * BN + STAGES * kSfCols;
    static constexpr uint32_t kTmemCols =
        kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128 : kColsUsed <= 256 ? 256 : 512;
    static_assert(kColsUsed <= 512, "TMEM budget");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    // split-K over a cluster of SPLIT CTAs: after the main loop the ring holds
    // the receive slots, then the send staging, of the column-ownership
    // reduction (4 warps x (SPLIT-1) slots of 32 rows x BN/SPLIT fp32 each)
    static constexpr uint32_t kSplitW = BN / SPLIT;
    static constexpr uint32_t kSplitSlotBytes = 32 * kSplitW * 4;
    static constexpr uint32_t kSplitSlots = 4 * (SPLIT - 1);
    static constexpr uint32_t kSplitSendOff = kSplitSlots * kSplitSlotBytes;
    static_assert(SPLIT == 1 || (ACC == 1 && kSplitW % 32 == 0 &&
                                 2 * kSplitSlots * kSplitSlotBytes <= STAGES * kStageBytes),
                  "split-K slots reuse the ring");
    // Split-K epilogue groups: warps 2-5, and (kSplitEH = 2, MXFP8) warps 0, 1, 6, 7,
    // idle once the main loop is done; the group of warp w sums and stores
    // columns [h*kSplitWH, (h+1)*kSplitWH) of each split's W in TMEM lane
    // quarter w % 4.  Both groups stage their stores in the ring, after the
    // receive slots and the send staging.
    static constexpr uint32_t kSplitEH =
        (KIND == kKindMXF8 && SPLIT > 1 && kSplitW >= 64 &&
         2 * kSplitSlots * kSplitSlotBytes + 8 * kEpiWarpBytes <= STAGES * kStageBytes)
            ? 2u : 1u;                       // the second group needs an 8th warp (MXFP8 CTAs only)
    static constexpr uint32_t kSplitWH = kSplitW / kSplitEH;
    static constexpr uint32_t kSplitSubBytes = 32 * kSplitWH * 4;    // one warp's rows of its kSplitWH columns
    static constexpr uint32_t kSplitEpi0Off = 2 * kSplitSlots * kSplitSlotBytes;
    static constexpr uint32_t kSplitEpi1Off = kSplitEpi0Off + 4 * kEpiWarpBytes;
    static_assert(kSplitWH % 32 == 0, "whole 32-column chunks per split and group");
    static_assert(SPLIT == 1 || kSplitEpi0Off + kSplitEH * 4 * kEpiWarpBytes <= STAGES * kStageBytes,
                  "split-K store staging in the ring");
    static constexpr uint32_t smem_bytes(uint32_t groups) { return 1024 + kTableOff + 8 * (groups + 1); }
    // fp16/bf16, BN 64, plain GEMMs whose B has the two-row view (b.rows2):
    // kRows2Slots staging slots of one k-block's even rows (32 x 128 bytes)
    // and odd rows (32 x 144 bytes, 8 bytes early), where the group table
    // would be
    static constexpr uint32_t kRows2Slots = 4;
    static constexpr uint32_t kRows2EvenBytes = 32 * 128;
    static constexpr uint32_t kRows2Slot = kRows2EvenBytes + 32 * 144;
    static constexpr uint32_t kRows2Off = (kTableOff + 127) & ~127u;
    static constexpr uint32_t smem_bytes_rows2() { return 1024 + kRows2Off + kRows2Slots * kRows2Slot; }
};

// Warp-wide wait: every lane polls the barrier itself and the result is made
// warp-uniform.  Measured on sm_103a, this is much cheaper for the warp's
// following work than one lane polling while the others wait at a warp
// barrier (an MMA loop waiting that way ran at a third of the tensor rate).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
    const bool ok = mbar_wait(bar, parity, ctl, where);
    return __all_sync(0xFFFFFFFFu, ok);
}

// What the scheduler needs, in registers.
struct SchedArgs {
    uint32_t M, N, swz_offset, swz_dir, mode, total_m;
    const PlainSched* ps;   // plain / batched: the host-prepared scheduler
};

struct TileInfo {
    uint32_t tag;      // batch index or group index
    uint32_t m, n;     // tile indices
    uint32_t m_act, n_act;
    uint32_t row0;     // first row of the tile in A / C (includes the group offset)
    uint32_t m_lim;    // rows of A that exist (loads past it read zeros)
};

// Task t -> tile of TM x BN (TM = 128 for one CTA, 256 for a CTA pair).
__device__ __forceinline__ TileInfo tile_info(const SchedArgs& sa, uint32_t t, uint32_t TM, uint32_t BN,
                                              const GroupTable& gt) {
    TileInfo ti;
    SwizzleSched s;
    if (sa.mode == kModeGrouped) {
        const uint32_t g = gt.find(t);
        const uint32_t mg = gt.row_off[g + 1] - gt.row_off[g];
        s.update(mg, sa.N, TM, BN, sa.swz_offset, sa.swz_dir);
        s.block_coord(t - gt.tile_off[g], ti.m, ti.n);
        s.actual_shape(ti.m, ti.n, ti.m_act, ti.n_act);
        ti.tag = g;
        ti.row0 = gt.row_off[g] + ti.m * TM;
        ti.m_lim = sa.total_m;
    } else {
        sa.ps->coord(t, ti.tag, ti.m, ti.n, ti.m_act, ti.n_act);
        ti.row0 = ti.m * TM;
        ti.m_lim = sa.M;
    }
    return ti;
}

// Grouped slice-M: one warp computes the exclusive prefix sums of rows and of
// tiles (tile_m x tile_n) over the groups into shared memory and stores the
// task count in *tiles_out; inconsistent sizes (a negative size, or more rows
// than total_m) give no tasks and raise the error word.
__device__ __forceinline__ void build_group_table(const GroupTable& gt, const int32_t* group_m, uint32_t G, uint32_t N,
                                                  uint32_t TM, uint32_t BN, uint32_t total_m, uint32_t* err,
                                                  uint32_t* tiles_out, uint32_t lane) {
    const uint32_t loops_n = (N + BN - 1) / BN;
    uint32_t row_carry = 0, tile_carry = 0, bad = 0;
    if (lane == 0) { gt.row_off[0] = 0; gt.tile_off[0] = 0; }
    for (uint32_t base = 0; base < G; base += 32) {
        const uint32_t g = base + lane;
        int32_t mg = g < G ? group_m[g] : 0;
        if (mg < 0) { bad = 1; mg = 0; }
        uint32_t rows = static_cast<uint32_t>(mg);
        uint32_t tiles = ((rows + TM - 1) / TM) * loops_n;
#pragma unroll
        for (uint32_t d = 1; d < 32; d <<= 1) {
            const uint32_t r = __shfl_up_sync(0xFFFFFFFFu, rows, d);
            const uint32_t tt = __shfl_up_sync(0xFFFFFFFFu, tiles, d);
            if (lane >= d) { rows += r; tiles += tt; }
        }
        if (g < G) {
            gt.row_off[g + 1] = row_carry + rows;
            gt.tile_off[g + 1] = tile_carry + tiles;
        }
        row_carry += __shfl_sync(0xFFFFFFFFu, rows, 31);
        tile_carry += __shfl_sync(0xFFFFFFFFu, tiles, 31);
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
        if (bad || row_carry > total_m) {
            *tiles_out = 0;
            if (blockIdx.x == 0) atomicOr(&err[0], kErrGroups);
        } else {
            *tiles_out = tile_carry;
        }
    }
}

// Fallback for operands TMA cannot fetch (pitch or base not 16-byte
// aligned).  Writes the exact shared-memory image a TMA load with 128-byte
// swizzle would: line L (128 bytes) at L*128, its 16-byte chunk c at
// ((c ^ (L % 8)) * 16); out-of-range elements are zero, like TMA's
// out-of-bounds fill.  The warp moves the tile in V-byte vectors (V = 16, 8,
// 4 or 2, the widest the operand's base and pitch allow): each lane first
// loads 8 vectors through L2 into registers (so 256 loads of the warp are in
// flight together), then stores them.  The stores are generic-proxy writes:
// the caller fences them for the async proxy before arriving on the stage
// barrier.  (A cp.async version of this loader issued each warp-wide copy in
// roughly 0.3 us when L1 is almost entirely carved out for the stage ring.)
template <uint32_t V>
struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<2> { using T = uint16_t; };

__device__ __forceinline__ uint4 ld_cg(const uint4* p) { return __ldcg(p); }
__device__ __forceinline__ uint2 ld_cg(const uint2* p) { return __ldcg(p); }
__device__ __forceinline__ uint32_t ld_cg(const uint32_t* p) { return __ldcg(p); }
__device__ __forceinline__ uint16_t ld_cg(const uint16_t* p) { return __ldcg(p); }

// The first n bytes at p (n < V, a multiple of the element size esize), zero
// above: the ragged end of a row, read element by element into two 64-bit
// halves (no dynamically indexed register array, which would live in local
// memory).
template <uint32_t V>
__device__ __forceinline__ typename VecT<V>::T ld_partial(const uint8_t* p, uint32_t n, uint32_t esize) {
    uint64_t lo = 0, hi = 0;
    for (uint32_t b = 0; b < n; b += esize) {
        const uint64_t x = esize == 1 ? static_cast<uint64_t>(__ldcg(reinterpret_cast<const unsigned char*>(p + b)))
                                      : static_cast<uint64_t>(__ldcg(reinterpret_cast<const uint16_t*>(p + b)));
        if (b < 8) lo |= x << (b * 8);
        else hi |= x << ((b - 8) * 8);
    }
    typename VecT<V>::T out;
    if constexpr (V == 16)
        out = make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32), static_cast<uint32_t>(hi),
                         static_cast<uint32_t>(hi >> 32));
    else if constexpr (V == 8) out = make_uint2(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32));
    else if constexpr (V == 4) out = static_cast<uint32_t>(lo);
    else out = static_cast<uint16_t>(lo);
    return out;
}

// Operands reaching this loader are 2-byte (fp16/bf16); the element size,
// the vector width and the layout are compile-time, so the per-vector index
// arithmetic is a few shifts and adds.
template <uint32_t V, bool MN>
__device__ __noinline__ static void load_tile_regs(uint8_t* dst, const uint8_t* base, int64_t ld, uint32_t lines,
                                                   uint32_t mn0, uint32_t mn_lim, uint32_t k0, uint32_t k_lim,
                                                   uint32_t lane) {
    using T = typename VecT<V>::T;
    constexpr uint32_t kEsize = 2;
    constexpr uint32_t kLineElems = kLine / kEsize;   // 64
    constexpr uint32_t vpl = kLine / V;               // vectors per 128-byte line
    constexpr uint32_t kBatch = 8;
    const uint32_t total = lines * vpl;
    const uint32_t byte_in_line = (lane % vpl) * V;   // the same for every vector of this lane (vpl divides 32)
    const uint32_t e_in_line = byte_in_line / kEsize;
    static_assert(32 % vpl == 0 || vpl % 32 == 0, "lane pattern");
#pragma unroll 1
    for (uint32_t i0 = 0; i0 < total; i0 += 32 * kBatch) {
        T tmp[kBatch];
        uint32_t off[kBatch];
#pragma unroll
        for (uint32_t u = 0; u < kBatch; ++u) {
            const uint32_t idx = i0 + u * 32 + lane;
            const uint32_t L = idx / vpl;
            const uint32_t bil = vpl <= 32 ? byte_in_line : (idx % vpl) * V;
            const uint32_t eil = vpl <= 32 ? e_in_line : bil / kEsize;
            uint32_t outer, outer_lim, e, inner_lim;
            if (!MN) {                    // line = one MN row, a k-block of K
                outer = mn0 + L;
                outer_lim = mn_lim;
                e = k0 + eil;
                inner_lim = k_lim;
            } else {                      // line = one k of a 64-element MN atom
                outer = k0 + (L % kLineElems);
                outer_lim = k_lim;
                e = mn0 + (L / kLineElems) * kLineElems + eil;
                inner_lim = mn_lim;
            }
            off[u] = idx < total ? L * kLine + ((((bil >> 4) ^ (L & 7u)) << 4) | (bil & 15u)) : 0xFFFFFFFFu;
            const uint32_t in_elems = (idx < total && outer < outer_lim && e < inner_lim) ? inner_lim - e : 0u;
            const uint32_t in_bytes = min(V, in_elems * kEsize);
            const uint8_t* src = base + (static_cast<int64_t>(outer) * ld + e) * kEsize;
            if (in_bytes == V) tmp[u] = ld_cg(reinterpret_cast<const T*>(src));
            else if (in_bytes) tmp[u] = ld_partial<V>(src, in_bytes, kEsize);
            else tmp[u] = T{};
        }
#pragma unroll
        for (uint32_t u = 0; u < kBatch; ++u)
            if (off[u] != 0xFFFFFFFFu) *reinterpret_cast<T*>(dst + off[u]) = tmp[u];
    }
}

// The same shared-memory image by cp.async (V = 4, 8 or 16): every vector of
// the tile is in flight at once, straight from L2 into shared memory, with
// out-of-range bytes zero-filled by the copy itself.  The caller follows
// with cp.async.mbarrier.arrive, so the stage's barrier completes when this
// lane's copies have landed (the MMA thread fences for the async proxy).
// Inlined: as a called function it took ~0.3 us of issue time per k-block.
template <uint32_t V, bool MN>
__device__ __forceinline__ static void load_tile_async(uint8_t* dst, const uint8_t* base, int64_t ld, uint32_t lines,
                                                       uint32_t mn0, uint32_t mn_lim, uint32_t k0, uint32_t k_lim,
                                                       uint32_t lane, uint32_t part, uint32_t nparts) {
    constexpr uint32_t kEsize = 2;
    constexpr uint32_t kLineElems = kLine / kEsize;   // 64
    constexpr uint32_t vpl = kLine / V;               // vectors per 128-byte line: 8, 16 or 32
    static_assert(32 % vpl == 0, "lane pattern");
    constexpr uint32_t kLinesPerPass = 32 / vpl;
    const uint32_t bil = (lane % vpl) * V;            // byte of this lane's vectors within their lines
    const uint32_t eil = bil / kEsize;
#pragma unroll 4
    for (uint32_t L = lane / vpl + part * kLinesPerPass; L < lines; L += nparts * kLinesPerPass) {
        uint32_t outer, outer_lim, e, inner_lim;
        if (!MN) {                    // line = one MN row, a k-block of K
            outer = mn0 + L;
            outer_lim = mn_lim;
            e = k0 + eil;
            inner_lim = k_lim;
        } else {                      // line = one k of a 64-element MN atom
            outer = k0 + (L % kLineElems);
            outer_lim = k_lim;
            e = mn0 + (L / kLineElems) * kLineElems + eil;
            inner_lim = mn_lim;
        }
        const uint32_t in_elems = (outer < outer_lim && e < inner_lim) ? inner_lim - e : 0u;
        const uint32_t in_bytes = min(V, in_elems * kEsize);
        const uint8_t* src = in_bytes ? base + (static_cast<int64_t>(outer) * ld + e) * kEsize : base;
        cp_async_v<V>(dst + L * kLine + ((((bil >> 4) ^ (L & 7u)) << 4) | (bil & 15u)), src, in_bytes);
    }
}

// Returns true when the copies went out asynchronously (the caller then
// arrives with cp.async.mbarrier.arrive), false when they were register
// loads and stores (2-byte vectors, which cp.async cannot copy).
__device__ __forceinline__ bool load_tile_plain(uint8_t* dst, const uint8_t* base, int64_t ld, uint32_t mn_major,
                                                uint32_t V, uint32_t esize, uint32_t lines, uint32_t mn0,
                                                uint32_t mn_lim, uint32_t k0, uint32_t k_lim, uint32_t lane,
                                                uint32_t part, uint32_t nparts) {
    (void)esize;   // always 2 here
    if (mn_major) {
        switch (V) {
            case 16: load_tile_async<16, true>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            case 8: load_tile_async<8, true>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            case 4: load_tile_async<4, true>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            default:
                if (part == 0) load_tile_regs<2, true>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane);
                return false;
        }
    } else {
        switch (V) {
            case 16: load_tile_async<16, false>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            case 8: load_tile_async<8, false>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            case 4: load_tile_async<4, false>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane, part, nparts); return true;
            default:
                if (part == 0) load_tile_regs<2, false>(dst, base, ld, lines, mn0, mn_lim, k0, k_lim, lane);
                return false;
        }
    }
}

// Issues the TMA loads of one operand tile: one box for K-contiguous
// operands, one box per 128-byte MN atom otherwise.
__device__ __forceinline__ void tma_tile(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, uint32_t mn_major,
                                         uint32_t rank3, uint32_t mn0, uint32_t rows, uint32_t k0, int32_t z,
                                         uint32_t bk_elems) {
    if (!mn_major) {
        if (rank3) tma_load_3d(dst, map, bar, k0, mn0, z);
        else tma_load_2d(dst, map, bar, k0, mn0);
    } else {
        for (uint32_t j = 0; j < rows / bk_elems; ++j) {
            uint8_t* d = dst + j * bk_elems * kLine;
            const int32_t x = mn0 + j * bk_elems;
            if (rank3) tma_load_3d(d, map, bar, x, k0, z);
            else tma_load_2d(d, map, bar, x, k0);
        }
    }
}

// Stores one 32 x 32 output chunk that a warp holds one row per lane (v[j] =
// column j as 32-bit data: fp32 bits converted to out_type, or with kOutS32 a
// raw int32).  The chunk goes through the warp's 4 KB staging buffer -- rows
// of 64 (16-bit) or 128 (32-bit) bytes whose 16-byte granules are XOR-swizzled
// by row, so the row-wise writes and the segment-wise reads are both free of
// bank conflicts -- and leaves as whole row segments: consecutive lanes store
// consecutive VEC-byte pieces of one row, so every store instruction writes
// full sectors.  Rows >= rows_valid and columns >= cols_valid are not written
// (both warp-uniform).  c0 addresses row 0, column 0 of the chunk; ld_bytes is
// the row pitch; VEC (at least the element size ESZ) divides c0's address and
// ld_bytes.  Everything but the data is compile-time, and every shared-memory
// read of the chunk is issued before the first global store: one warp runs
// this alone, so a loop of dependent address arithmetic would cost it
// hundreds of cycles per pass.
template <uint32_t ESZ, uint32_t VEC>
__device__ __forceinline__ void store_chunk_t(uint8_t* stage, uint32_t out_type, uint8_t* c0, int64_t ld_bytes,
                                              uint32_t rows_valid, uint32_t cols_valid, const uint32_t (&v)[32],
                                              uint32_t lane) {
    using T = typename VecT<VEC>::T;
    constexpr uint32_t kRowBytes = 32u * ESZ;
    constexpr uint32_t kLanesPerRow = kRowBytes / VEC;   // 4 .. 32
    constexpr uint32_t kRowsPerPass = 32u / kLanesPerRow;
    constexpr uint32_t kPasses = 32u / kRowsPerPass;
    static_assert(VEC >= ESZ && kLanesPerRow <= 32, "vector width");
    if (ESZ == 2) {
        uint32_t p[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (out_type == kOutF16) {
                const __half2 h = __floats2half2_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                p[j] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __nv_bfloat162 h =
                    __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                p[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        uint8_t* rowp = stage + lane * 64u;
        const uint32_t f = (lane >> 1) & 3u;
#pragma unroll
        for (uint32_t g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(rowp + ((g ^ f) << 4)) = make_uint4(p[4 * g], p[4 * g + 1], p[4 * g + 2], p[4 * g + 3]);
    } else {
        uint8_t* rowp = stage + lane * 128u;
        const uint32_t f = lane & 7u;
#pragma unroll
        for (uint32_t g = 0; g < 8; ++g)
            *reinterpret_cast<uint4*>(rowp + ((g ^ f) << 4)) = make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    }
    __syncwarp();
    const uint32_t row_in_pass = lane / kLanesPerRow;
    const uint32_t byte_in_row = (lane % kLanesPerRow) * VEC;
    const uint32_t valid_bytes = cols_valid * ESZ;
    T val[kPasses];
#pragma unroll
    for (uint32_t q = 0; q < kPasses; ++q) {
        const uint32_t r = q * kRowsPerPass + row_in_pass;
        const uint32_t f = ESZ == 4 ? (r & 7u) : ((r >> 1) & 3u);
        val[q] = *reinterpret_cast<const T*>(stage + r * kRowBytes + ((((byte_in_row >> 4) ^ f) << 4) | (byte_in_row & 15u)));
    }
    uint8_t* dst = c0 + static_cast<int64_t>(row_in_pass) * ld_bytes + byte_in_row;
    const int64_t step = static_cast<int64_t>(kRowsPerPass) * ld_bytes;
    if (byte_in_row + VEC <= valid_bytes) {
#pragma unroll
        for (uint32_t q = 0; q < kPasses; ++q) {
            if (q * kRowsPerPass + row_in_pass < rows_valid) *reinterpret_cast<T*>(dst) = val[q];
            dst += step;
        }
    } else if (byte_in_row < valid_bytes) {
        // the ragged end of the rows: element by element
#pragma unroll 1
        for (uint32_t q = 0; q < kPasses; ++q) {
            const uint32_t r = q * kRowsPerPass + row_in_pass;
            if (r < rows_valid) {
                const uint32_t f = ESZ == 4 ? (r & 7u) : ((r >> 1) & 3u);
                const uint8_t* src = stage + r * kRowBytes + ((((byte_in_row >> 4) ^ f) << 4) | (byte_in_row & 15u));
                for (uint32_t b = 0; b < valid_bytes - byte_in_row; b += ESZ) {
                    if (ESZ == 4) *reinterpret_cast<uint32_t*>(dst + b) = *reinterpret_cast<const uint32_t*>(src + b);
                    else *reinterpret_cast<uint16_t*>(dst + b) = *reinterpret_cast<const uint16_t*>(src + b);
                }
            }
            dst += step;
        }
    }
    __syncwarp();
}

__device__ __forceinline__ void store_chunk_coalesced(uint8_t* stage, uint32_t out_type, uint32_t vec, uint8_t* c0,
                                                      int64_t ld_bytes, uint32_t rows_valid, uint32_t cols_valid,
                                                      const uint32_t (&v)[32], uint32_t lane) {
    if (out_type == kOutF32 || out_type == kOutS32) {
        if (vec >= 16) store_chunk_t<4, 16>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
        else if (vec == 8) store_chunk_t<4, 8>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
        else store_chunk_t<4, 4>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
    } else {
        if (vec >= 16) store_chunk_t<2, 16>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
        else if (vec == 8) store_chunk_t<2, 8>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
        else if (vec == 4) store_chunk_t<2, 4>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
        else store_chunk_t<2, 2>(stage, out_type, c0, ld_bytes, rows_valid, cols_valid, v, lane);
    }
}

// SPLIT > 1: split-K over clusters of SPLIT CTAs, one output tile per cluster
// (cluster rank = split); the partial tiles are summed through distributed
// shared memory by column ownership (see the end of the kernel).
template <uint32_t BN, uint32_t STAGES, uint32_t ACC, uint32_t KIND, uint32_t EPI, uint32_t SPLIT = 1>
__global__ void __launch_bounds__(threads_for<KIND>(), 1) gemm_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = GemmLayout<BN, STAGES, ACC, KIND, SPLIT>;
    static_assert(SPLIT == 1 || (EPI == kEpiStore && (SPLIT == 2 || SPLIT == 4)), "split-K: plain stores, 2 or 4");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(EPI == kEpiStore || BN == 128, "dequant epilogue keeps 128 int32 per thread");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // ---- arguments into registers, once
    const uint64_t t_entry = globaltimer_ns();
    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m, &prm.g.ps};
    const uint32_t N = prm.g.N, K = prm.g.K, mode = prm.g.mode, esize = prm.g.esize;
    const uint32_t num_kb = prm.g.num_kb, chunk_kb = prm.g.chunk_kb, G = prm.g.G;
    const uint32_t a_tma = prm.g.a.use_tma, b_tma = prm.g.b.use_tma;
    const uint32_t a_mn = prm.g.a.mn_major, b_mn = prm.g.b.mn_major;
    const uint32_t a_rank3 = prm.g.a.tma_rank == 3, b_rank3 = prm.g.b.tma_rank == 3;
    uint32_t* const err = prm.g.err;
    uint64_t* const tl = prm.g.timeline ? prm.g.timeline + static_cast<uint64_t>(blockIdx.x) * 64 : nullptr;
    const uint32_t bk_elems = kLine / esize;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + ACC;
    uint64_t* drain = bars + 2 * STAGES + 2 * ACC;
    uint64_t* raw_full = bars + 2 * STAGES + 2 * ACC + 1;
    uint64_t* recv = bars + 2 * STAGES + 2 * ACC + 5;
    uint64_t* rows2_free = recv;                          // two-row view B (never split): 4 slot barriers
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    uint32_t* tiles_smem = misc + 2;

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    // B through the two-row view (plain fp16/bf16, BN 64, A by TMA): warp
    // kBWarp loads it by TMA into staging and rewrites it into the ring
    const bool b_rows2 = KIND == kKindF16 && BN == 64 && prm.g.b.rows2 != 0;
    const bool lanes_copy = KIND == kKindMXF8 || !(a_tma && (b_tma || b_rows2));
    const bool lanes_copy_ops = !(a_tma && (b_tma || b_rows2));   // an operand goes through the load/store units
    // Operands TMA cannot fetch go through the load/store unit, whose
    // throughput per warp is the limit: for the CTA's first tile the epilogue
    // warps, idle until its accumulator is ready, copy too (six warps in all).
    // One accumulator chunk per tile, so that no epilogue is due before the
    // first tile's copies are issued.
    const bool copy_helpers = KIND == kKindF16 && EPI == kEpiStore && lanes_copy_ops && prm.g.chunk_kb >= num_kb;

    GroupTable gt;
    gt.G = G;
    gt.tile_off = reinterpret_cast<uint32_t*>(smem + Lay::kTableOff);
    gt.row_off = gt.tile_off + (mode == kModeGrouped ? G + 1 : 0);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            // 1 arrival from the issuing lane (+ TMA bytes), plus one per lane
            // when lanes also copy (MXFP8 scale factors, non-TMA operands)
            // (MXFP8 with scale TMA: the A thread and one arrival of the scale warp)
            // (fp16/bf16 with an operand TMA cannot fetch: warps 0 and kBWarp both
            // copy, and with copy helpers so do warps 2-5 -- on later tiles warp 0
            // arrives for them)
            // (B through the two-row view: the A thread, and four from the rewriting warps)
            mbar_init(&full[s], (KIND == kKindMXF8 && prm.g.sf_tma) ? 2u
                                : lanes_copy ? (KIND == kKindF16 && lanes_copy_ops ? (copy_helpers ? 193u : 65u) : 33u)
                                : b_rows2    ? 5u
                                             : 1u);
            mbar_init(&empty[s], 1);
        }
        for (uint32_t a = 0; a < ACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        for (uint32_t r = 0; r < 4; ++r) mbar_init(&raw_full[r], 1);   // MXFP8: 2 raw slots; two-row B: 4
        // (two-row view B: recv[0..3] are the staging slots' rows2_free, four arrivals each)
        for (uint32_t o = 0; o < 8; ++o) mbar_init(&recv[o], (b_rows2 && o < 4) ? 4u : 1u);
        *abort_flag = 0;
        *tiles_smem = prm.g.total_tiles;
        fence_barrier_init();
        // split-K: each epilogue warp's receive barrier expects SPLIT-1 partials
        if (SPLIT > 1)
            for (uint32_t o = 0; o < 4 * Lay::kSplitEH; ++o)
                mbar_arrive_expect_tx(&recv[o], (SPLIT - 1) * Lay::kSplitSubBytes);
    }
    if (warp == 0 && lane == 0) {
        if (a_tma) prefetch_tmap(&prm.tmap_a);
        if (b_tma) prefetch_tmap(&prm.tmap_b);
        if (b_rows2) {
            prefetch_tmap(&prm.tmap_sfa);
            prefetch_tmap(&prm.tmap_sfb);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Lay::kTmemCols);
        tmem_relinquish();
    }
    // small problems: the epilogue warps (idle until the first accumulator is
    // ready) pull the operands into L2 while the previous kernel finishes (a
    // prefetch reads nothing into the SM, and L2 is coherent with whatever
    // that kernel still writes)
    if ((SPLIT == 1 || KIND == kKindF16) && warp >= 2 && warp < 6) prefetch_operands(prm.g, threadIdx.x - 64, 128);
    // set-up above reads no global memory into the SM: it overlaps the previous kernel
    griddep_wait();
    griddep_launch_dependents();
    if (mode == kModeGrouped && warp == 2)
        build_group_table(gt, prm.g.group_m, G, N, kBM, BN, sa.total_m, err, tiles_smem, lane);
    __syncwarp();                                    // reconverge lane-0 set-up branches first
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t total_tiles = *tiles_smem;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    if (tl && threadIdx.x == 0) { tl[0] = globaltimer_ns(); tl[55] = t_entry; }
    // tiles of this CTA and its k-block range: persistent stride, or (split-K)
    // the cluster's one tile and this split's share of K, in whole 4-k-block
    // groups when the MXFP8 scale factors come by TMA
    const uint32_t split = SPLIT > 1 ? cluster_rank() : 0u;
    const uint32_t t_first = SPLIT > 1 ? cluster_id_x() : blockIdx.x;
    const uint32_t t_step = SPLIT > 1 ? total_tiles : gridDim.x;
    uint32_t kb_lo = 0, kb_hi = num_kb;
    if (SPLIT > 1) {
        const uint32_t gran = (KIND == kKindMXF8 && prm.g.sf_tma) ? 4u : 1u;
        const uint32_t units = (num_kb + gran - 1) / gran;
        kb_lo = min(num_kb, (split * units / SPLIT) * gran);
        kb_hi = min(num_kb, ((split + 1) * units / SPLIT) * gran);
    }
    const bool has_k = kb_hi > kb_lo;
    // ShuffleK (fp16/bf16): task t's K loop starts at k-block kb_lo + t % (kb_hi - kb_lo)
    const uint32_t nk_span = kb_hi - kb_lo;
    auto shuffle_rot = [&](uint32_t t) -> uint32_t {
        return (KIND == kKindF16 && prm.g.shuffle_k && nk_span) ? t % nk_span : 0u;
    };
    auto shuffled = [&](uint32_t kb, uint32_t rot) -> uint32_t {
        const uint32_t kx = kb + rot;
        return kx < kb_hi ? kx : kx - nk_span;
    };
    bool acc_ok = true;                                  // split-K: this CTA's partial is complete

    // ------------------------------ copy helpers (first tile only) --
    auto copy_first_tile_as_helper = [&]() {
        if (!copy_helpers || t_first >= total_tiles) return;
        // parts 2-5 of the six-way split of every k-block's copies (warps
        // 0 and kBWarp take parts 0 and 1); TMA, where an operand allows
        // it, stays with the load thread
        const TileInfo ti = tile_info(sa, t_first, kBM, BN, gt);
        const uint32_t n0 = ti.n * BN;
        const uint32_t rot = shuffle_rot(t_first);
        const uint32_t a_vec = prm.g.a.vec_bytes, b_vec = prm.g.b.vec_bytes;
        const int64_t a_bs = prm.g.a.batch_stride, b_bs = prm.g.b.batch_stride;
        uint32_t stage = 0, phase = 0, issued = 0;
        for (uint32_t kb = kb_lo; kb < kb_hi; ++kb) {
            if (issued >= STAGES && !warp_wait(&empty[stage], phase ^ 1u, ctl, 1)) break;
            uint8_t* sa_s = smem + stage * Lay::kStageBytes;
            uint8_t* sb_s = sa_s + Lay::kABytes;
            const uint32_t k0 = shuffled(kb, rot) * bk_elems;
            bool async_only = true;
            if (!a_tma && !load_tile_plain(sa_s, prm.g.a.ptr + (a_rank3 ? ti.tag * a_bs * esize : 0), prm.g.a.ld,
                                           a_mn, a_vec, esize, kBM, ti.row0, ti.m_lim, k0, K, lane, warp, 6u))
                async_only = false;
            if (!b_tma && !load_tile_plain(sb_s,
                                           prm.g.b.ptr + ((mode != kModePlain && b_bs != 0) ? ti.tag * b_bs * esize : 0),
                                           prm.g.b.ld, b_mn, b_vec, esize, BN, n0, N, k0, K, lane, warp, 6u))
                async_only = false;
            if (!async_only) fence_proxy_async_smem();
            cp_async_arrive_noinc(&full[stage]);
            if (tl && warp == 2 && lane == 0 && issued < 7) tl[8 + issued] = globaltimer_ns();
            ++issued;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        __syncwarp();
    };

    // ------------------------------- B through the two-row view (warp kBWarp) --
    // A 16-bit MN-major B whose pitch is 8 bytes off a multiple of 16 has no
    // tensor map, but pairs of rows do: in a view with rows of 2*ld elements,
    // a k-block's 32 even rows are one 64 x 32 box at x = n0 and its 32 odd
    // rows one 72 x 32 box at x = ld + n0 - 4 (the nearest 16-byte boundary,
    // 8 bytes early).  Lane 0 of warp kBWarp keeps four k-blocks of these
    // boxes in flight in four staging slots (raw_full[] completes them).  A
    // k-block is rewritten into the ring's B slot in the SW128 layout (line L
    // = k-row L, 16-byte granule g at g ^ (L % 8)), fenced for the async proxy
    // and arrived on the stage's full barrier, which expects the A thread (with
    // A's bytes) and four arrivals: for the CTA's first tile the four epilogue
    // warps (idle until its accumulator is ready) each rewrite 16 lines and
    // arrive, and arrive on the slot's rows2_free barrier so that the slot is
    // refilled only once all four have read it; for later tiles warp kBWarp
    // rewrites all 64 lines and arrives for four.
    const uint32_t rows2_nk = kb_hi - kb_lo;
    const uint32_t rows2_items =
        (t_first < total_tiles ? (total_tiles - t_first + t_step - 1) / t_step : 0u) * rows2_nk;
    // lines [line0, line0 + 4 * reps) of item i's staging slot into the ring
    auto rows2_convert = [&](uint32_t i, uint32_t line0, auto reps_c) {
        constexpr uint32_t kReps = decltype(reps_c)::value;     // granules per lane
        const uint8_t* even = smem + Lay::kRows2Off + (i % Lay::kRows2Slots) * Lay::kRows2Slot;
        const uint8_t* odd = even + Lay::kRows2EvenBytes;
        uint8_t* dst = smem + (i % STAGES) * Lay::kStageBytes + Lay::kABytes;
        const uint32_t g = lane & 7u;
        // batches of up to 8 granules per lane, all loads of a batch before its
        // stores (interleaved, every store waits for the loads before it)
#pragma unroll
        for (uint32_t b0 = 0; b0 < kReps; b0 += 8) {
            constexpr uint32_t kB = kReps < 8 ? kReps : 8;
            uint2 lo[kB], hi[kB];
#pragma unroll
            for (uint32_t r = 0; r < kB; ++r) {
                const uint32_t L = line0 + (lane >> 3) + 4 * (b0 + r);
                const uint8_t* src = (L & 1u) ? odd + (L >> 1) * 144 + 8 + g * 16 : even + (L >> 1) * 128 + g * 16;
                lo[r] = *reinterpret_cast<const uint2*>(src);
                hi[r] = *reinterpret_cast<const uint2*>(src + 8);
            }
#pragma unroll
            for (uint32_t r = 0; r < kB; ++r) {
                const uint32_t L = line0 + (lane >> 3) + 4 * (b0 + r);
                *reinterpret_cast<uint4*>(dst + L * kLine + ((g ^ (L & 7u)) << 4)) =
                    make_uint4(lo[r].x, lo[r].y, hi[r].x, hi[r].y);
            }
        }
        // the ring's bytes -> the MMA's reads; the slot's reads -> the next
        // TMA writes into it
        fence_proxy_async_smem();
        __syncwarp();
    };
    // warps 2-5: the first tile's k-blocks, 16 lines each
    auto rows2_help_first_tile = [&]() {
        if (!b_rows2) return;
        const uint32_t n = min(rows2_nk, rows2_items);
        for (uint32_t i = 0; i < n; ++i) {
            if (!warp_wait(&raw_full[i % Lay::kRows2Slots], (i / Lay::kRows2Slots) & 1u, ctl, 9)) break;
            if (i >= STAGES && !warp_wait(&empty[i % STAGES], ((i / STAGES) & 1u) ^ 1u, ctl, 1)) break;
            rows2_convert(i, (warp - 2) * 16, std::integral_constant<uint32_t, 4>{});
            if (lane == 0) {
                mbar_arrive(&full[i % STAGES]);
                mbar_arrive(&rows2_free[i % Lay::kRows2Slots]);
            }
            __syncwarp();
        }
    };
    // warp kBWarp: issues every item's boxes; rewrites the items after the first tile
    auto load_b_rows2 = [&]() {
        constexpr uint32_t kSlots = Lay::kRows2Slots;
        const uint32_t nk = rows2_nk, items = rows2_items;
        const int32_t ld = static_cast<int32_t>(prm.g.b.ld);
        uint32_t t_cached = 0xFFFFFFFFu;
        TileInfo ti_cached{};
        auto issue = [&](uint32_t i) {                   // lane 0: item i into slot i % kSlots
            const uint32_t t = t_first + (i / nk) * t_step;
            if (t != t_cached) { ti_cached = tile_info(sa, t, kBM, BN, gt); t_cached = t; }
            const int32_t n0 = static_cast<int32_t>(ti_cached.n * BN);
            const int32_t y = static_cast<int32_t>(shuffled(kb_lo + i % nk, shuffle_rot(t)) * bk_elems / 2);
            uint8_t* slot = smem + Lay::kRows2Off + (i % kSlots) * Lay::kRows2Slot;
            mbar_arrive_expect_tx(&raw_full[i % kSlots], Lay::kRows2Slot);   // both boxes, out-of-range parts included
            tma_load_2d(slot, &prm.tmap_sfa, &raw_full[i % kSlots], n0, y);
            tma_load_2d(slot + Lay::kRows2EvenBytes, &prm.tmap_sfb, &raw_full[i % kSlots], ld + n0 - 4, y);
        };
        if (lane == 0)
            for (uint32_t i = 0; i < kSlots && i < items; ++i) issue(i);
        __syncwarp();
        uint32_t i = 0;
        for (; i < items; ++i) {
            if (i < nk) {
                // the helpers rewrite it; refill its slot once they all have
                if (i + kSlots < items && !warp_wait(&rows2_free[i % kSlots], (i / kSlots) & 1u, ctl, 10)) break;
            } else {
                if (!warp_wait(&raw_full[i % kSlots], (i / kSlots) & 1u, ctl, 9)) break;
                if (i >= STAGES && !warp_wait(&empty[i % STAGES], ((i / STAGES) & 1u) ^ 1u, ctl, 1)) break;
                rows2_convert(i, 0u, std::integral_constant<uint32_t, 16>{});
                if (lane == 0) mbar_arrive_cnt(&full[i % STAGES], 4u);
            }
            if (lane == 0) {
                if (tl && i < 7) tl[8 + i] = globaltimer_ns();
                if (i + kSlots < items) issue(i + kSlots);
            }
            __syncwarp();
        }
        if (lane == 0)                                   // staging copies still in flight land before exit
            for (uint32_t j = i; j < items && j < i + kSlots; ++j)
                mbar_wait_drain(&raw_full[j % kSlots], (j / kSlots) & 1u, ctl.timeout_ns);
    };

    constexpr uint32_t kBWarp = b_warp_for<KIND>();
    if (warp == 0 || (KIND == kKindMXF8 && warp == kScaleWarp) ||
        (warp == kBWarp && ((lanes_copy_ops || b_rows2) ? KIND == kKindF16 : lane == 0))) {
        // ------------------------------------------------------ producer --
        const uint8_t* a_ptr = prm.g.a.ptr;
        const uint8_t* b_ptr = prm.g.b.ptr;
        const int64_t a_ld = prm.g.a.ld, b_ld = prm.g.b.ld;
        const int64_t a_bs = prm.g.a.batch_stride, b_bs = prm.g.b.batch_stride;
        const uint32_t a_vec = prm.g.a.vec_bytes, b_vec = prm.g.b.vec_bytes;
        const uint8_t* sfa = prm.g.sfa;
        const uint8_t* sfb = prm.g.sfb;
        const uint32_t sf_ld = prm.g.sf_ld;
        const uint32_t tx = (a_tma ? Lay::kABytes : 0u) + (b_tma ? Lay::kBBytes : 0u);
        // Roles of the load warps:
        // - Both operands through TMA: lane 0 of warp 0 issues the A loads and
        //   is the one arrival on full[] (expecting the bytes of A and B), lane
        //   0 of warp kBWarp issues the B loads.  A B load may land before the A
        //   thread's expect_tx: the transaction count goes negative meanwhile and
        //   the missing arrival keeps the phase open.  A thread running such a
        //   loop alone issues a k-block in about half the time of one that shares
        //   a warp-synchronous loop.
        // - B through the two-row view: warp kBWarp as a whole (load_b_rows2).
        // - An operand TMA cannot fetch: warps 0 and kBWarp copy it with their
        //   lanes (the epilogue warps help on the first tile); lane 0 of warp 0
        //   also issues the TMA half of a mixed stage.
        // - MXFP8: the scale warp copies the scale factors.
        const bool copy_split = KIND == kKindF16 && lanes_copy_ops;   // warps 0 and kBWarp share the copies
        const bool tma_thread = (warp == 0 && lane == 0) || (warp == kBWarp && lane == 0 && !copy_split);
        const bool warp_copies = (KIND == kKindMXF8) ? (warp == kScaleWarp)
                                                     : ((warp == 0 || (copy_split && warp == kBWarp)) && lanes_copy);
        const uint32_t copy_part = warp == kBWarp ? 1u : 0u, copy_parts = copy_split ? 2u : 1u;
        if (b_rows2 && warp == kBWarp) {
            if constexpr (KIND == kKindF16 && BN == 64) load_b_rows2();
        } else if (tma_thread && !warp_copies) {
            const bool is_a = warp == 0;
            const bool simple = !a_mn && !b_mn && !a_rank3 && !b_rank3;
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t t = t_first; ok && t < total_tiles; t += t_step) {
                if (tl && is_a && issued == 0) tl[56] = globaltimer_ns();
                const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
                const uint32_t n0 = ti.n * BN;
                const int32_t zc = static_cast<int32_t>(ti.tag);
                if (tl && is_a && issued == 0) tl[57] = globaltimer_ns();
                if (simple) {
                    // both operands K-contiguous, 2-D maps: one box per k-block
                    const CUtensorMap* map = is_a ? &prm.tmap_a : &prm.tmap_b;
                    const uint32_t dst_off = is_a ? 0u : Lay::kABytes;
                    const int32_t row = is_a ? static_cast<int32_t>(ti.row0) : static_cast<int32_t>(n0);
                    const uint32_t rot = shuffle_rot(t);
                    for (uint32_t kb = kb_lo; kb < kb_hi; ++kb) {
                        // the ring starts empty: only a stage being reused is waited for
                        if (issued >= STAGES && !mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                        uint8_t* st = smem + stage * Lay::kStageBytes;
                        const int32_t k0 = static_cast<int32_t>(shuffled(kb, rot) * bk_elems);
                        if (is_a) mbar_arrive_expect_tx(&full[stage], tx);
                        tma_load_2d(st + dst_off, map, &full[stage], k0, row);
                        if (tl && is_a && issued < 15) tl[1 + issued] = globaltimer_ns();
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    continue;
                }
                const uint32_t rot = shuffle_rot(t);
                for (uint32_t kb = kb_lo; kb < kb_hi; ++kb) {
                    if (issued >= STAGES && !mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    const uint32_t k0 = shuffled(kb, rot) * bk_elems;
                    if (is_a) {
                        mbar_arrive_expect_tx(&full[stage], tx);
                        tma_tile(&prm.tmap_a, sa_s, &full[stage], a_mn, a_rank3, ti.row0, kBM, k0, zc, bk_elems);
                    } else {
                        tma_tile(&prm.tmap_b, sa_s + Lay::kABytes, &full[stage], b_mn, b_rank3, n0, BN, k0, zc,
                                 bk_elems);
                    }
                    if (tl && is_a && issued < 15) tl[1 + issued] = globaltimer_ns();
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                uint32_t s = stage, ph = phase;
                const uint32_t pending = issued < STAGES ? issued : STAGES;
                for (uint32_t i = 0; i < pending; ++i) {
                    if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                    mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
                }
            }
        } else if (warp_copies && KIND == kKindMXF8 && prm.g.sf_tma) {
            // Scale factors by TMA: every 4 k-blocks lane 0 loads 16 bytes of
            // each of the tile's rows (the codes of 4 k-blocks) into one of two
            // raw slots, one group ahead; per k-block the warp rewrites them into
            // the stage's lines in the order tcgen05.cp 32x128b.warpx4 expects
            // (16-byte line l holds rows l, l+32, l+64, l+96, 4 bytes each) and
            // makes one arrival on the stage's full barrier.  Only this warp
            // touches the raw slots, so they need no empty barrier.
            constexpr uint32_t kRawA = Lay::kRawRowsA * 16u;
            constexpr uint32_t raw_bytes = Lay::kRawSlotBytes;
            uint32_t stage = 0, phase = 0;
            uint32_t rg = 0, cg = 0;                     // raw groups issued / consumed (slot = n % 2)
            bool ok = true;
            for (uint32_t t = t_first; ok && t < total_tiles; t += t_step) {
                const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
                const int32_t n0 = static_cast<int32_t>(ti.n * BN);
                const uint32_t ngroups = (kb_hi + 3) / 4;      // groups are absolute: kb / 4
                auto issue = [&](uint32_t g) {
                    uint8_t* slot = smem + Lay::kRawOff + (rg & 1u) * raw_bytes;
                    fence_proxy_async_smem();            // earlier reads of this slot before the new writes
                    mbar_arrive_expect_tx(&raw_full[rg & 1u], raw_bytes);
                    tma_load_2d(slot, &prm.tmap_sfa, &raw_full[rg & 1u], static_cast<int32_t>(g * 16), ti.row0);
                    tma_load_2d(slot + kRawA, &prm.tmap_sfb, &raw_full[rg & 1u], static_cast<int32_t>(g * 16), n0);
                    ++rg;
                };
                if (lane == 0 && has_k) issue(kb_lo / 4);
                for (uint32_t kb = kb_lo; kb < kb_hi; ++kb) {
                    const uint32_t j = kb & 3u;
                    if (j == 0) {
                        if (lane == 0 && kb / 4 + 1 < ngroups) issue(kb / 4 + 1);
                        if (!warp_wait(&raw_full[cg & 1u], (cg >> 1) & 1u, ctl, 6)) { ok = false; break; }
                    }
                    if (!warp_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                    const uint8_t* raw = smem + Lay::kRawOff + (cg & 1u) * raw_bytes + lane * 16u + j * 4u;
                    uint8_t* sfa_s = smem + Lay::kSfOff + stage * Lay::kSfStageBytes;
                    uint8_t* sfb_s = sfa_s + Lay::kSfaBytes;
                    *reinterpret_cast<uint4*>(sfa_s + lane * 16u) =
                        make_uint4(*reinterpret_cast<const uint32_t*>(raw), *reinterpret_cast<const uint32_t*>(raw + 512),
                                   *reinterpret_cast<const uint32_t*>(raw + 1024),
                                   *reinterpret_cast<const uint32_t*>(raw + 1536));
#pragma unroll
                    for (uint32_t h = 0; h < BN / 128; ++h) {
                        const uint8_t* rb = raw + kRawA + h * 2048u;
                        *reinterpret_cast<uint4*>(sfb_s + h * 512 + lane * 16u) =
                            make_uint4(*reinterpret_cast<const uint32_t*>(rb), *reinterpret_cast<const uint32_t*>(rb + 512),
                                       *reinterpret_cast<const uint32_t*>(rb + 1024),
                                       *reinterpret_cast<const uint32_t*>(rb + 1536));
                    }
                    fence_proxy_async_smem();            // generic writes -> tcgen05.cp's reads
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[stage]);
                    if (j == 3 || kb + 1 == kb_hi) ++cg;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && lane == 0) {
                // let the raw scale copies in flight land before the CTA exits
                while (cg < rg) {
                    mbar_wait_drain(&raw_full[cg & 1u], (cg >> 1) & 1u, ctl.timeout_ns);
                    ++cg;
                }
            }
        } else if (warp_copies) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t t = t_first; ok && t < total_tiles; t += t_step) {
                const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
                const uint32_t n0 = ti.n * BN;
                const int32_t zc = static_cast<int32_t>(ti.tag);
                const uint32_t rot = shuffle_rot(t);
                const bool helped = copy_helpers && t == t_first;
                const uint32_t parts = helped ? 6u : copy_parts;
                for (uint32_t kb = kb_lo; kb < kb_hi; ++kb) {
                    // the ring starts empty: only a stage being reused is waited for
                    if (issued >= STAGES && !warp_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    uint8_t* sb_s = sa_s + Lay::kABytes;
                    const uint32_t k0 = shuffled(kb, rot) * bk_elems;
                    if (KIND == kKindMXF8) {
                        // scale factors for this k-block, written straight into the
                        // order tcgen05.cp 32x128b.warpx4 expects: 16-byte line r%32
                        // holds rows r%32, +32, +64, +96 (4 bytes each = the 4
                        // E8M0 codes of the k-block's four 32-element sub-blocks)
                        uint8_t* sfa_s = smem + Lay::kSfOff + stage * Lay::kSfStageBytes;
                        uint8_t* sfb_s = sfa_s + Lay::kSfaBytes;
#pragma unroll
                        for (uint32_t i = 0; i < 4; ++i) {
                            const uint32_t r = lane + 32 * i;
                            const bool v = ti.row0 + r < ti.m_lim;
                            const uint8_t* src = v ? sfa + static_cast<int64_t>(ti.row0 + r) * sf_ld + kb * 4 : sfa;
                            cp_async_4(sfa_s + (lane * 4 + i) * 4, src, v ? 4u : 0u);
                        }
#pragma unroll
                        for (uint32_t h = 0; h < (BN >= 128 ? BN / 128 : 0u); ++h) {
#pragma unroll
                            for (uint32_t i = 0; i < 4; ++i) {
                                const uint32_t r = 128 * h + lane + 32 * i;
                                const bool v = n0 + r < N;
                                const uint8_t* src = v ? sfb + static_cast<int64_t>(n0 + r) * sf_ld + kb * 4 : sfb;
                                cp_async_4(sfb_s + h * 512 + (lane * 4 + i) * 4, src, v ? 4u : 0u);
                            }
                        }
                        cp_async_arrive_noinc(&full[stage]);
                    } else {
                        // operands TMA cannot fetch: cp.async where the vectors
                        // allow it (the lane's arrival fires when its copies
                        // land), else register copies, fenced before the arrival
                        bool async_only = true;
                        if (!a_tma && !load_tile_plain(sa_s, a_ptr + (a_rank3 ? ti.tag * a_bs * esize : 0), a_ld,
                                                       a_mn, a_vec, esize, kBM, ti.row0, ti.m_lim, k0, K, lane,
                                                       copy_part, parts))
                            async_only = false;
                        if (!b_tma && !load_tile_plain(sb_s,
                                                       b_ptr + ((mode != kModePlain && b_bs != 0) ? ti.tag * b_bs * esize : 0),
                                                       b_ld, b_mn, b_vec, esize, BN, n0, N, k0, K, lane, copy_part, parts))
                            async_only = false;
                        // register-copied bytes -> the MMA's reads.  Not after
                        // cp.async alone: the fence would wait for the copies to
                        // land, serialising the k-blocks; the MMA warp fences
                        // for them once the stage's barrier has completed.
                        if (!async_only) fence_proxy_async_smem();
                        cp_async_arrive_noinc(&full[stage]);
                        if (tl && warp == 0 && lane == 0 && issued < 7) tl[1 + issued] = globaltimer_ns();
                        // the helpers' 128 arrivals, on the tiles they do not copy
                        if (copy_helpers && !helped && warp == 0 && lane == 0) mbar_arrive_cnt(&full[stage], 128u);
                        if (tma_thread) {                // the TMA half of a mixed stage
                            mbar_arrive_expect_tx(&full[stage], tx);
                            if (a_tma)
                                tma_tile(&prm.tmap_a, sa_s, &full[stage], a_mn, a_rank3, ti.row0, kBM, k0, zc, bk_elems);
                            if (b_tma)
                                tma_tile(&prm.tmap_b, sb_s, &full[stage], b_mn, b_rank3, n0, BN, k0, zc, bk_elems);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && tma_thread) {
                uint32_t s = stage, ph = phase;
                const uint32_t pending = issued < STAGES ? issued : STAGES;
                for (uint32_t i = 0; i < pending; ++i) {
                    if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                    mbar_wait_drain(&full[s], ph, ctl.timeout_ns);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer --
        const uint32_t umma_k_bytes_mn = (32u / esize) * kLine;   // MN-major: UMMA_K rows of 128 B
        const uint32_t a_lbo = a_mn ? bk_elems * kLine : 16u;
        const uint32_t b_lbo = b_mn ? bk_elems * kLine : 16u;
        const uint32_t a_step = a_mn ? umma_k_bytes_mn : 32u;
        const uint32_t b_step = b_mn ? umma_k_bytes_mn : 32u;
        const uint32_t idesc = idesc_f16(prm.g.ab_fmt, a_mn, b_mn, kBM, BN);
        const uint32_t smem_base = smem_u32(smem);
        const uint32_t sf_tma = prm.g.sf_tma;
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, mma_kb = 0;
        bool ok = true, any_mma = false;
        const uint32_t nchunks = SPLIT > 1 ? (has_k ? 1u : 0u) : (num_kb + chunk_kb - 1) / chunk_kb;
        // the whole warp runs the loop (waits are warp-wide); the elected lane
        // (lane 0) issues every MMA, scale copy and commit
        for (uint32_t t = t_first; ok && t < total_tiles; t += t_step) {
            for (uint32_t c = 0; ok && c < nchunks; ++c) {
                const uint32_t kb_begin = SPLIT > 1 ? kb_lo : c * chunk_kb;
                const uint32_t kb_end = SPLIT > 1 ? kb_hi : min(num_kb, kb_begin + chunk_kb);
                if (!warp_wait(&tempty[acc], acc_phase ^ 1u, ctl, 2)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                    if (!warp_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
                    tc_fence_after();
                    // bytes written by cp.async (MXFP8 scale factors, operands
                    // TMA cannot fetch) need a proxy fence before tcgen05 reads
                    // them (every other writer fences before it arrives)
                    if ((KIND == kKindMXF8 && !sf_tma) || lanes_copy_ops) fence_proxy_async_smem();
                    if (elect_one()) {
                        if (tl && mma_kb < 16) tl[16 + mma_kb] = globaltimer_ns();
                        const uint32_t sa_addr = smem_base + stage * Lay::kStageBytes;
                        const uint32_t sb_addr = sa_addr + Lay::kABytes;
                        const uint64_t adesc = smem_desc(sa_addr, a_lbo, 1024, kSwizzle128B);
                        const uint64_t bdesc = smem_desc(sb_addr, b_lbo, 1024, kSwizzle128B);
                        if (KIND == kKindMXF8) {
                            const uint32_t sf_col = ACC * BN + stage * Lay::kSfCols;
                            const uint32_t sfa_addr = smem_base + Lay::kSfOff + stage * Lay::kSfStageBytes;
                            tmem_cp_32x128b_warpx4(tmem_base + sf_col, smem_desc(sfa_addr, 0, 128, kSwizzleNone));
#pragma unroll
                            for (uint32_t h = 0; h < (BN >= 128 ? BN / 128 : 0u); ++h)
                                tmem_cp_32x128b_warpx4(tmem_base + sf_col + 4 + 4 * h,
                                                       smem_desc(sfa_addr + Lay::kSfaBytes + h * 512, 0, 128, kSwizzleNone));
#pragma unroll
                            for (uint32_t kk = 0; kk < 4; ++kk)
                                umma_mxf8(d_tmem, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4),
                                          idesc_mxf8(kBM, BN, kk), tmem_base + sf_col, tmem_base + sf_col + 4,
                                          (kb > kb_begin || kk > 0) ? 1u : 0u);
                        } else {
#pragma unroll
                            for (uint32_t kk = 0; kk < 4; ++kk)
                                umma_f16(d_tmem, adesc + ((kk * a_step) >> 4), bdesc + ((kk * b_step) >> 4), idesc,
                                         (kb > kb_begin || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty[stage]);
                    }
                    __syncwarp();
                    ++mma_kb;
                    any_mma = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (elect_one()) umma_commit(&tfull[acc]);
                __syncwarp();
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
        }
        if (lane == 0 && !ok && any_mma) {
            // every tcgen05 op issued so far must finish before TMEM is freed
            umma_commit(drain);
            mbar_wait_drain(drain, 0, ctl.timeout_ns);
        }
    } else if (SPLIT > 1 && warp >= 2 && warp < 6) {
        // ------------------------------------- split-K epilogue, part 1 --
        // this CTA's partial is final once its MMAs are done; the exchange
        // follows the cluster barrier below
        copy_first_tile_as_helper();
        if (has_k && t_first < total_tiles) acc_ok = warp_wait(&tfull[0], 0, ctl, 4);
    } else if (warp >= 2 && warp < 6) {
        copy_first_tile_as_helper();
        if constexpr (KIND == kKindF16 && BN == 64) rows2_help_first_tile();
        // ----------------------------------------------------- epilogue --
        const uint32_t q = warp & 3u;            // TMEM lane quarter of this warp
        const uint32_t r = q * 32 + lane;        // tile row of this thread
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec, acc_vec = prm.g.acc_vec;
        uint8_t* const epi_stage = smem + Lay::kEpiOff + q * kEpiWarpBytes;
        uint8_t* const C = prm.g.C;
        const int64_t ldc = prm.g.ldc, c_bs = prm.g.c_batch_stride;
        const float* scale_a = prm.g.scale_a;
        const float* scale_b = prm.g.scale_b;
        int32_t* const acc_out = prm.g.acc_out;
        uint32_t* const trace = prm.g.trace;
        const uint32_t trace_cap = prm.g.trace_cap;
        const uint32_t nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
        const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
        uint32_t acc = 0, acc_phase = 0, ep_tile = 0;
        bool ok = true;
        for (uint32_t t = t_first; ok && t < total_tiles; t += t_step) {
            const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
            if (trace && warp == 2 && lane == 0) {
                if (t < trace_cap) {
                    uint32_t* tr = trace + static_cast<uint64_t>(t) * 5;
                    tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
                } else {
                    atomicOr(&err[0], kErrTraceOverflow);
                }
            }
            const bool row_ok = r < ti.m_act;
            const uint32_t grow = ti.row0 + r;
            const uint32_t rows_valid = ti.m_act > q * 32 ? min(32u, ti.m_act - q * 32) : 0u;   // warp-uniform
            const int64_t cbase = mode == kModeBatched ? static_cast<int64_t>(ti.tag) * c_bs : 0;
            // row q*32 of the tile (lane 0's row)
            uint8_t* const cwarp = C + (cbase + static_cast<int64_t>(ti.row0 + q * 32) * ldc) * csize;
            const uint32_t n0 = ti.n * BN;
            int32_t run[EPI == kEpiDequant ? BN : 1];
            if (EPI == kEpiDequant) {
#pragma unroll
                for (uint32_t j = 0; j < (EPI == kEpiDequant ? BN : 1); ++j) run[j] = 0;
            }
            for (uint32_t c = 0; c < nchunks; ++c) {
                if (!warp_wait(&tfull[acc], acc_phase, ctl, 4)) { ok = false; break; }
                tc_fence_after();
                if (tl && warp == 2 && lane == 0 && c == 0 && ep_tile < 8) tl[32 + ep_tile] = globaltimer_ns();
                const uint32_t taddr = tmem_base + ((q * 32) << 16) + acc * BN;
                if (EPI == kEpiStore) {
#pragma unroll 1
                    for (uint32_t cc = 0; cc < BN / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + cc * 32, v);
                        if (rows_valid && cc * 32 < ti.n_act)
                            store_chunk_coalesced(epi_stage, c_type, c_vec,
                                                  cwarp + static_cast<int64_t>(n0 + cc * 32) * csize, ldc * csize,
                                                  rows_valid, min(32u, ti.n_act - cc * 32), v, lane);
                    }
                } else {
#pragma unroll
                    for (uint32_t cc = 0; cc < BN / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + cc * 32, v);
#pragma unroll
                        for (uint32_t j = 0; j < 32; ++j)
                            run[(EPI == kEpiDequant ? cc * 32 + j : 0)] += __float2int_rn(__uint_as_float(v[j]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;
            if (tl && warp == 2 && lane == 0 && ep_tile < 8) tl[40 + ep_tile] = globaltimer_ns();
            ++ep_tile;
            if (EPI == kEpiDequant && rows_valid) {
                const float sa_row = row_ok ? scale_a[grow] : 0.f;
#pragma unroll
                for (uint32_t cc = 0; cc < BN / 32; ++cc) {
                    if (cc * 32 >= ti.n_act) break;
                    const uint32_t col0 = n0 + cc * 32;
                    const uint32_t nv = min(32u, ti.n_act - cc * 32);
                    uint32_t v[32];
#pragma unroll
                    for (uint32_t j = 0; j < 32; ++j) {
                        const float sb = j < nv ? __ldg(scale_b + col0 + j) : 0.f;
                        v[j] = __float_as_uint(static_cast<float>(run[(EPI == kEpiDequant ? cc * 32 + j : 0)]) * sa_row * sb);
                    }
                    store_chunk_coalesced(epi_stage, c_type, c_vec, cwarp + static_cast<int64_t>(col0) * csize,
                                          ldc * csize, rows_valid, nv, v, lane);
                    if (acc_out) {
#pragma unroll
                        for (uint32_t j = 0; j < 32; ++j)
                            v[j] = static_cast<uint32_t>(run[(EPI == kEpiDequant ? cc * 32 + j : 0)]);
                        uint8_t* awarp = reinterpret_cast<uint8_t*>(acc_out + static_cast<int64_t>(ti.row0 + q * 32) * ldc + col0);
                        store_chunk_coalesced(epi_stage, kOutS32, acc_vec, awarp, ldc * 4, rows_valid, nv, v, lane);
                    }
                }
            }
        }
    }

    if (SPLIT > 1) {
        // ------------------------------------- split-K epilogue, part 2 --
        // Every CTA of the cluster is past its main loop (its ring is idle)
        // once this barrier completes.  Split g finishes columns [g*W,
        // (g+1)*W) of the tile.  Every epilogue warp stages, for each other
        // split g, its 32 rows of its group's half (or all) of g's columns in
        // the ring (row per lane, 16-byte granules XOR-swizzled by row) and
        // bulk-copies them into a receive slot of CTA g, completing on that
        // CTA's receive barrier of the same warp; it then adds the SPLIT-1
        // partials it received to its own rows of its own columns, rounds once
        // and stores.
        __syncwarp();
        tc_fence_before();
        cluster_sync();                                  // also orders this CTA's own warps
        tc_fence_after();
        const bool epi_main = warp >= 2 && warp < 6;
        if ((epi_main || (Lay::kSplitEH == 2 && (warp < 2 || warp >= 6))) && t_first < total_tiles) {
            constexpr uint32_t W = Lay::kSplitW, WH = Lay::kSplitWH, EH = Lay::kSplitEH;
            constexpr uint32_t kSlot = Lay::kSplitSubBytes;
            const uint32_t q = warp & 3u;
            const uint32_t h = epi_main ? 0u : 1u;       // column group of this warp
            const uint32_t qh = q * EH + h;              // receive barrier and slot group
            const uint32_t taddr = tmem_base + ((q * 32) << 16);
            // warps 2-5 waited for the accumulator before the barrier; the
            // second group relies on that wait (no abort recorded since)
            const bool own_valid = (epi_main ? acc_ok : *abort_flag == 0) && has_k;   // else zeros
            uint32_t gi = 0;
#pragma unroll 1
            for (uint32_t g = 0; g < SPLIT; ++g) {
                if (g == split) continue;
                uint8_t* stage_rows = smem + Lay::kSplitSendOff + (qh * (SPLIT - 1) + gi) * kSlot;
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
                fence_proxy_async_smem();                // generic writes -> the bulk copy's reads
                __syncwarp();
                if (lane == 0) {
                    const uint32_t slot = qh * (SPLIT - 1) + (split < g ? split : split - 1);
                    const uint32_t dst = map_to_cta(smem_u32(smem + slot * kSlot), g);
                    const uint32_t bar = map_to_cta(smem_u32(&recv[qh]), g);
                    bulk_copy_to_cluster(dst, stage_rows, kSlot, bar);
                    bulk_commit_group();
                }
                ++gi;
            }
            const bool got = warp_wait(&recv[qh], 0, ctl, 5);
            const TileInfo ti = tile_info(sa, t_first, kBM, BN, gt);
            const uint8_t* slots = smem + qh * (SPLIT - 1) * kSlot + lane * (WH * 4);
            const uint32_t rows_valid = ti.m_act > q * 32 ? min(32u, ti.m_act - q * 32) : 0u;
            const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
            const uint32_t csize = c_type == kOutF32 ? 4u : 2u;
            const int64_t ldc = prm.g.ldc;
            uint8_t* const cwarp = prm.g.C + static_cast<int64_t>(ti.row0 + q * 32) * ldc * csize;
            uint8_t* const epi_stage = smem + (h ? Lay::kSplitEpi1Off : Lay::kSplitEpi0Off) + q * kEpiWarpBytes;
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
                    for (uint32_t si = 0; si < SPLIT - 1; ++si) {
#pragma unroll
                        for (uint32_t gg = 0; gg < 8; ++gg) {
                            const uint32_t granule = (cc * 8 + gg) ^ (lane & 7u);
                            const uint4 x = *reinterpret_cast<const uint4*>(slots + si * kSlot + granule * 16);
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
            if (lane == 0) bulk_wait_read_all();         // the ring may not be left while being read
            if (prm.g.trace && split == 0 && q == 0 && h == 0 && lane == 0 && t_first < prm.g.trace_cap) {
                uint32_t* tr = prm.g.trace + static_cast<uint64_t>(t_first) * 5;
                tr[0] = ti.tag; tr[1] = ti.m; tr[2] = ti.n; tr[3] = ti.m_act; tr[4] = ti.n_act;
            }
        }
        __syncwarp();
        tc_fence_before();
        cluster_sync();                                  // no CTA leaves while a peer may still touch it
    }
    if (tl && lane == 0 && warp <= 2) tl[48 + warp] = globaltimer_ns();
    // single-lane roles leave their warps diverged: reconverge every warp
    // first, so that the block barrier counts each warp once (split tiles
    // have just passed the cluster barrier, which orders every warp already)
    __syncwarp();
    tc_fence_before();
    if (SPLIT == 1) __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Lay::kTmemCols);
    }
}

}  // namespace bst
