// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks the task indices t = blockIdx.x, blockIdx.x + grid,
// ... ; each task index is turned into an output tile by the block-swizzle
// scheduler (sched.cuh, "Block Scheduler Code Explained" sections 4-7).
// Roles inside the CTA (192 threads):
//   warp 0     producer: per k-block waits for a free shared-memory stage and
//              fills it (TMA, or cp.async for operands TMA cannot take; MXFP8
//              scale factors by cp.async) -- the counterpart of the GM->L1
//              copies of "Block Dispatch Policies" (MmadAtlasA2Preload /
//              PreloadAsync: the producer runs ahead across tile and group
//              boundaries, i.e. inter-block and inter-group preloading).
//   warp 1     MMA issuer: one thread issues tcgen05.mma into a TMEM
//              accumulator, releasing each stage with tcgen05.commit.
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

#include "ptx.cuh"
#include "sched.cuh"

namespace bst {

enum : uint32_t { kKindF16 = 0, kKindMXF8 = 1 };
enum : uint32_t { kEpiStore = 0, kEpiDequant = 1 };
enum : uint32_t { kModePlain = 0, kModeBatched = 1, kModeGrouped = 2 };
enum : uint32_t { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2 };

constexpr uint32_t kBM = 128;          // tile rows = TMEM lanes
constexpr uint32_t kLine = 128;        // bytes per k-block line
constexpr uint32_t kNumThreads = 192;   // warps: 0 TMA, 1 MMA, 2-5 epilogue
constexpr uint32_t kScaleWarp = 6;      // MXFP8 only: a 7th warp copies scale factors
template <uint32_t KIND>
constexpr uint32_t threads_for() { return KIND == 1 ? kNumThreads + 32 : kNumThreads; }
constexpr uint32_t kMaxGroups = 1024;

struct OperandDesc {
    const uint8_t* ptr;
    int64_t ld;            // elements
    int64_t batch_stride;  // elements
    uint32_t mn_major;     // 1: the M (or N) index is contiguous
    uint32_t use_tma;
    uint32_t vec_bytes;    // cp.async / plain-load vector width when !use_tma
    uint32_t tma_rank;     // 2, or 3 when the tensor map has a batch/group dimension
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
    uint32_t c_vec;         // 16-byte vector stores allowed for whole 32-column chunks
    const float* scale_a;
    const float* scale_b;
    int32_t* acc_out;
    const uint8_t* sfa;
    const uint8_t* sfb;
    uint32_t sf_ld;         // bytes per row of sfa / sfb (K / 32)
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

struct GemmParams {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;
    GemmArgs g;
};

template <uint32_t BN, uint32_t STAGES, uint32_t ACC, uint32_t KIND>
struct GemmLayout {
    static constexpr uint32_t kABytes = kBM * kLine;
    static constexpr uint32_t kBBytes = BN * kLine;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kSfaBytes = KIND == kKindMXF8 ? 512u : 0u;
    static constexpr uint32_t kSfbBytes = KIND == kKindMXF8 ? BN * 4u : 0u;
    static constexpr uint32_t kSfStageBytes = kSfaBytes + kSfbBytes;
    static constexpr uint32_t kSfOff = STAGES * kStageBytes;
    static constexpr uint32_t kBarOff = kSfOff + STAGES * kSfStageBytes;
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * ACC + 1;
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
    static constexpr uint32_t smem_bytes(uint32_t groups) { return 1024 + kTableOff + 8 * (groups + 1); }
};

// One lane of the warp waits on the barrier (the others would only add
// shared-memory traffic); the warp then re-converges, with the memory
// ordering of __syncwarp, and every lane gets the same verdict, so a timeout
// never splits the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
    uint32_t ok = 1;
    if ((threadIdx.x & 31u) == 0) ok = mbar_wait(bar, parity, ctl, where) ? 1u : 0u;
    __syncwarp();
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// What the scheduler needs, in registers.
struct SchedArgs {
    uint32_t M, N, swz_offset, swz_dir, mode, total_m;
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
        s.update(sa.M, sa.N, TM, BN, sa.swz_offset, sa.swz_dir);
        ti.tag = s.batch_idx(t);
        s.block_coord(t, ti.m, ti.n);
        s.actual_shape(ti.m, ti.n, ti.m_act, ti.n_act);
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
// out-of-bounds fill.  Vectors of 4-16 bytes go through cp.async (zero-fill
// past the edge) and complete on the stage barrier through the caller's
// cp.async.mbarrier.arrive; 2-byte vectors (odd pitches) use plain loads and
// stores and the caller fences them for the async proxy.
__device__ __noinline__ static void load_tile_plain(uint8_t* dst, const uint8_t* base, int64_t ld, uint32_t mn_major,
                                                    uint32_t V, uint32_t esize, uint32_t lines, uint32_t mn0,
                                                    uint32_t mn_lim, uint32_t k0, uint32_t k_lim, uint32_t lane) {
    const uint32_t line_elems = kLine / esize;
    const uint32_t vpl = kLine / V;
    const uint32_t total = lines * vpl;
    for (uint32_t idx = lane; idx < total; idx += 32) {
        const uint32_t L = idx / vpl;
        const uint32_t byte_in_line = (idx % vpl) * V;
        uint32_t outer, outer_lim, inner0, inner_lim;
        if (!mn_major) {              // line = one MN row, a k-block of K
            outer = mn0 + L;
            outer_lim = mn_lim;
            inner0 = k0;
            inner_lim = k_lim;
        } else {                      // line = one k of a 64/128-element MN atom
            outer = k0 + L % line_elems;
            outer_lim = k_lim;
            inner0 = mn0 + (L / line_elems) * line_elems;
            inner_lim = mn_lim;
        }
        const uint32_t e = inner0 + byte_in_line / esize;
        uint8_t* d = dst + L * kLine + ((((byte_in_line >> 4) ^ (L & 7u)) << 4) | (byte_in_line & 15u));
        const bool row_in = outer < outer_lim;
        const uint32_t in_elems = (row_in && e < inner_lim) ? inner_lim - e : 0u;
        const uint32_t in_bytes = min(V, in_elems * esize);
        const uint8_t* src = in_bytes ? base + (static_cast<int64_t>(outer) * ld + e) * esize : base;
        if (V >= 4) {
            cp_async_n(d, src, V, in_bytes);
        } else {
            uint16_t v = 0;
            if (in_bytes) v = __ldg(reinterpret_cast<const uint16_t*>(src));
            *reinterpret_cast<uint16_t*>(d) = v;
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

// Stores 32 consecutive fp32 accumulator columns of one output row.
__device__ __forceinline__ void store_row_chunk(uint32_t c_type, uint32_t c_vec, uint8_t* row_ptr, uint32_t col0,
                                                uint32_t n_valid, const uint32_t (&v)[32]) {
    if (c_type == kOutF32) {
        float* out = reinterpret_cast<float*>(row_ptr) + col0;
        if (c_vec && n_valid >= 32) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<uint4*>(out + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
#pragma unroll
            for (uint32_t j = 0; j < 32; ++j)
                if (j < n_valid) out[j] = __uint_as_float(v[j]);
        }
        return;
    }
    uint32_t packed[16];
    if (c_type == kOutF16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            __half2 h = __floats2half2_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            packed[j] = *reinterpret_cast<uint32_t*>(&h);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            packed[j] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    uint16_t* out = reinterpret_cast<uint16_t*>(row_ptr) + col0;
    if (c_vec && n_valid >= 32) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<uint4*>(out + 2 * j) = make_uint4(packed[j], packed[j + 1], packed[j + 2], packed[j + 3]);
    } else {
#pragma unroll
        for (uint32_t j = 0; j < 32; ++j)
            if (j < n_valid) out[j] = static_cast<uint16_t>(j & 1 ? packed[j >> 1] >> 16 : packed[j >> 1] & 0xFFFFu);
    }
}

template <uint32_t BN, uint32_t STAGES, uint32_t ACC, uint32_t KIND, uint32_t EPI>
__global__ void __launch_bounds__(threads_for<KIND>(), 1) gemm_kernel(const __grid_constant__ GemmParams prm) {
    using Lay = GemmLayout<BN, STAGES, ACC, KIND>;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(EPI == kEpiStore || BN == 128, "dequant epilogue keeps 128 int32 per thread");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // ---- arguments into registers, once
    const uint64_t t_entry = globaltimer_ns();
    const SchedArgs sa{prm.g.M, prm.g.N, prm.g.swz_offset, prm.g.swz_dir, prm.g.mode, prm.g.total_m};
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
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    uint32_t* tiles_smem = misc + 2;

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const bool lanes_copy = KIND == kKindMXF8 || !(a_tma && b_tma);

    GroupTable gt;
    gt.G = G;
    gt.tile_off = reinterpret_cast<uint32_t*>(smem + Lay::kTableOff);
    gt.row_off = gt.tile_off + (mode == kModeGrouped ? G + 1 : 0);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            // 1 arrival from the issuing lane (+ TMA bytes), plus one per lane
            // when lanes also copy (MXFP8 scale factors, non-TMA operands)
            mbar_init(&full[s], lanes_copy ? 33u : 1u);
            mbar_init(&empty[s], 1);
        }
        for (uint32_t a = 0; a < ACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *tiles_smem = prm.g.total_tiles;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (a_tma) prefetch_tmap(&prm.tmap_a);
        if (b_tma) prefetch_tmap(&prm.tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Lay::kTmemCols);
        tmem_relinquish();
    }
    if (mode == kModeGrouped && warp == 2)
        build_group_table(gt, prm.g.group_m, G, N, kBM, BN, sa.total_m, err, tiles_smem, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t total_tiles = *tiles_smem;
    const WaitCtl ctl{abort_flag, prm.g.timeout_ns, err};
    if (tl && threadIdx.x == 0) { tl[0] = globaltimer_ns(); tl[55] = t_entry; }

    if (warp == 0 || (KIND == kKindMXF8 && warp == kScaleWarp)) {
        // ------------------------------------------------------ producer --
        const uint8_t* a_ptr = prm.g.a.ptr;
        const uint8_t* b_ptr = prm.g.b.ptr;
        const int64_t a_ld = prm.g.a.ld, b_ld = prm.g.b.ld;
        const int64_t a_bs = prm.g.a.batch_stride, b_bs = prm.g.b.batch_stride;
        const uint32_t a_vec = prm.g.a.vec_bytes, b_vec = prm.g.b.vec_bytes;
        const uint8_t* sfa = prm.g.sfa;
        const uint8_t* sfb = prm.g.sfb;
        const uint32_t sf_ld = prm.g.sf_ld;
        const bool plain_stores = (!a_tma && a_vec < 4) || (!b_tma && b_vec < 4);
        const uint32_t tx = (a_tma ? Lay::kABytes : 0u) + (b_tma ? Lay::kBBytes : 0u);
        // The TMA thread runs a loop of its own that contains no warp-synchronous
        // operation: mixing it with the warp-wide copy loop (whose waits end in
        // __syncwarp / shfl.sync) made every iteration pay for reconvergence
        // bookkeeping, and a tight single-thread loop issues a k-block in about
        // half the time.  Lanes copy only for the MXFP8 scale factors (their own
        // warp) and for operands TMA cannot fetch (warp 0, which then also
        // carries the TMA issue).
        const bool tma_thread = (warp == 0 && lane == 0);
        const bool warp_copies = (KIND == kKindMXF8) ? (warp == kScaleWarp) : (warp == 0 && lanes_copy);
        if (tma_thread && !warp_copies) {
            const bool simple = !a_mn && !b_mn && !a_rank3 && !b_rank3;
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                if (tl && issued == 0) tl[56] = globaltimer_ns();
                const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
                const uint32_t n0 = ti.n * BN;
                const int32_t zc = static_cast<int32_t>(ti.tag);
                if (tl && issued == 0) tl[57] = globaltimer_ns();
                if (simple) {
                    // both operands K-contiguous, 2-D maps: one box each per k-block
                    for (uint32_t kb = 0; kb < num_kb; ++kb) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                        uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                        const int32_t k0 = static_cast<int32_t>(kb * bk_elems);
                        mbar_arrive_expect_tx(&full[stage], tx);
                        tma_load_2d(sa_s, &prm.tmap_a, &full[stage], k0, ti.row0);
                        tma_load_2d(sa_s + Lay::kABytes, &prm.tmap_b, &full[stage], k0, n0);
                        if (tl && issued < 15) tl[1 + issued] = globaltimer_ns();
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    continue;
                }
                for (uint32_t kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    const uint32_t k0 = kb * bk_elems;
                    mbar_arrive_expect_tx(&full[stage], tx);
                    tma_tile(&prm.tmap_a, sa_s, &full[stage], a_mn, a_rank3, ti.row0, kBM, k0, zc, bk_elems);
                    tma_tile(&prm.tmap_b, sa_s + Lay::kABytes, &full[stage], b_mn, b_rank3, n0, BN, k0, zc, bk_elems);
                    if (tl && issued < 15) tl[1 + issued] = globaltimer_ns();
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
        } else if (warp_copies) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const TileInfo ti = tile_info(sa, t, kBM, BN, gt);
                const uint32_t n0 = ti.n * BN;
                const int32_t zc = static_cast<int32_t>(ti.tag);
                for (uint32_t kb = 0; kb < num_kb; ++kb) {
                    if (!warp_wait(&empty[stage], phase ^ 1u, ctl, 1)) { ok = false; break; }
                    uint8_t* sa_s = smem + stage * Lay::kStageBytes;
                    uint8_t* sb_s = sa_s + Lay::kABytes;
                    const uint32_t k0 = kb * bk_elems;
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
                        if (!a_tma)
                            load_tile_plain(sa_s, a_ptr + (a_rank3 ? ti.tag * a_bs * esize : 0), a_ld, a_mn, a_vec,
                                            esize, kBM, ti.row0, ti.m_lim, k0, K, lane);
                        if (!b_tma)
                            load_tile_plain(sb_s,
                                            b_ptr + ((mode != kModePlain && b_bs != 0) ? ti.tag * b_bs * esize : 0),
                                            b_ld, b_mn, b_vec, esize, BN, n0, N, k0, K, lane);
                        if (plain_stores) {
                            cp_async_wait_all();         // the other operand may have used cp.async
                            fence_proxy_async_smem();
                            mbar_arrive(&full[stage]);
                        } else {
                            cp_async_arrive_noinc(&full[stage]);
                        }
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
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, mma_kb = 0;
        bool ok = true, any_mma = false;
        const uint32_t nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
        // one thread issues every MMA (a single-lane loop, see the producer)
        for (uint32_t t = blockIdx.x; lane == 0 && ok && t < total_tiles; t += gridDim.x) {
            for (uint32_t c = 0; ok && c < nchunks; ++c) {
                const uint32_t kb_begin = c * chunk_kb;
                const uint32_t kb_end = min(num_kb, kb_begin + chunk_kb);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ctl, 2)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait(&full[stage], phase, ctl, 3)) { ok = false; break; }
                    tc_fence_after();
                    // stages written by cp.async / plain stores need a proxy
                    // fence before tcgen05 reads them
                    if (lanes_copy) fence_proxy_async_smem();
                    {
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
                    ++mma_kb;
                    any_mma = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
            }
        }
        if (lane == 0 && !ok && any_mma) {
            // every tcgen05 op issued so far must finish before TMEM is freed
            umma_commit(drain);
            mbar_wait_drain(drain, 0, ctl.timeout_ns);
        }
    } else if (warp >= 2 && warp < 6) {
        // ----------------------------------------------------- epilogue --
        prefetch_operands(prm.g, threadIdx.x - 64, 128);
        const uint32_t q = warp & 3u;            // TMEM lane quarter of this warp
        const uint32_t r = q * 32 + lane;        // tile row of this thread
        const uint32_t c_type = prm.g.c_type, c_vec = prm.g.c_vec;
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
        for (uint32_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
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
            const int64_t cbase = mode == kModeBatched ? static_cast<int64_t>(ti.tag) * c_bs : 0;
            uint8_t* crow = C + (cbase + static_cast<int64_t>(grow) * ldc) * csize;
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
                        if (row_ok && cc * 32 < ti.n_act)
                            store_row_chunk(c_type, c_vec, crow, n0 + cc * 32, ti.n_act - cc * 32, v);
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
            if (EPI == kEpiDequant && row_ok) {
                const float sa_row = scale_a[grow];
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
                    store_row_chunk(c_type, c_vec, crow, col0, nv, v);
                    if (acc_out) {
                        int32_t* arow = acc_out + static_cast<int64_t>(grow) * ldc + col0;
                        if (c_vec && nv == 32) {
#pragma unroll
                            for (uint32_t j = 0; j < 32; j += 4)
                                *reinterpret_cast<int4*>(arow + j) =
                                    make_int4(run[(EPI == kEpiDequant ? cc * 32 + j : 0)],
                                              run[(EPI == kEpiDequant ? cc * 32 + j + 1 : 0)],
                                              run[(EPI == kEpiDequant ? cc * 32 + j + 2 : 0)],
                                              run[(EPI == kEpiDequant ? cc * 32 + j + 3 : 0)]);
                        } else {
#pragma unroll
                            for (uint32_t j = 0; j < 32; ++j)
                                if (j < nv) arow[j] = run[(EPI == kEpiDequant ? cc * 32 + j : 0)];
                        }
                    }
                }
            }
        }
    }

    if (tl && lane == 0 && warp <= 2) tl[48 + warp] = globaltimer_ns();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Lay::kTmemCols);
    }
}

}  // namespace bst
