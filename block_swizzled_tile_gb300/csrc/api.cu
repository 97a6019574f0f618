// C-ABI entry points of include/bst.h: argument validation, TMA tensor-map
// construction, tile/grid selection and kernel launch.  No entry point
// allocates memory or synchronises (except bst_check_async).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "bst.h"
#include "internal.h"

namespace bst {

// Per-device error word: [0] flags (kErr*), [1] block, [2] where, [3] spare.
__device__ uint32_t g_err_word[4];

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    uint32_t sms = 0;
    uint32_t max_smem = 0;
    uint32_t* err = nullptr;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
thread_local uint64_t t_timeout_ns = 0;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The device whose primary context this host thread has made current (-1:
// none yet).  cudaGetDevice binds no context, and a thread that has made no
// other runtime call would reach the driver's tensor-map encoder without one.
thread_local int t_bound_dev = -1;

bst_status device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BST_ERR_CUDA;
    if (t_bound_dev != dev) {
        if (cudaSetDevice(dev) != cudaSuccess) return BST_ERR_CUDA;   // makes its primary context current
        t_bound_dev = dev;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return BST_ERR_CUDA;
        void* err = nullptr;
        if (cudaGetSymbolAddress(&err, g_err_word) != cudaSuccess) return BST_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sms = static_cast<uint32_t>(sms);
        d.max_smem = static_cast<uint32_t>(smem);
        d.err = static_cast<uint32_t*>(err);
        d.ready = true;
    }
    out = d;
    return d.supported ? BST_OK : BST_ERR_UNSUPPORTED;
}

bool encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

uint32_t dtype_bytes(bst_dtype t) {
    switch (t) {
        case BST_F16: case BST_BF16: return 2;
        case BST_E4M3: case BST_S8: return 1;
        case BST_F32: case BST_S32: return 4;
    }
    return 0;
}

bool out_code(bst_dtype t, uint32_t& code) {
    if (t == BST_F16) code = kOutF16;
    else if (t == BST_BF16) code = kOutBF16;
    else if (t == BST_F32) code = kOutF32;
    else return false;
    return true;
}

uint64_t timeout_ns() { return t_timeout_ns ? t_timeout_ns : kDefaultTimeoutNs; }

struct Sched {
    uint32_t offset = 1, dir = 0, tile_n = 0, tile_m = 0, num_ctas = 0, split_k = 0, shuffle_k = 0, dynamic = 0;
    uint32_t* trace = nullptr;
    uint64_t* timeline = nullptr;
};

bst_status read_sched(const bst_sched* s, Sched& out) {
    if (!s) return BST_OK;
    if (s->swizzle_offset < 1 || s->swizzle_direction > 1) return BST_ERR_INVALID_ARG;
    if (s->tile_n != 0 && s->tile_n != 64 && s->tile_n != 128 && s->tile_n != 256) return BST_ERR_INVALID_ARG;
    if (s->tile_m != 0 && s->tile_m != 128 && s->tile_m != 256) return BST_ERR_INVALID_ARG;
    if (s->split_k > 4 || s->split_k == 3) return BST_ERR_INVALID_ARG;
    if (s->shuffle_k > 1 || s->dynamic > 1) return BST_ERR_INVALID_ARG;
    if (s->dynamic && s->num_ctas) return BST_ERR_INVALID_ARG;            // the grid is one cluster per task
    if (s->dynamic && s->split_k >= 2) return BST_ERR_UNSUPPORTED;
    if (s->dynamic && s->tile_m == 128) return BST_ERR_UNSUPPORTED;        // CTA-pair tiles only
    out.shuffle_k = s->shuffle_k;
    out.dynamic = s->dynamic;
    out.offset = s->swizzle_offset;
    out.dir = s->swizzle_direction;
    out.tile_n = s->tile_n;
    out.tile_m = s->dynamic ? 256u : s->tile_m;
    out.split_k = s->split_k;
    out.num_ctas = s->num_ctas;
    out.trace = s->trace;
    out.timeline = s->timeline;
    return BST_OK;
}

// CTA pairs to launch: a persistent grid of at most one pair per two SMs (or
// num_ctas / 2), or -- with dynamic tasks -- one cluster per task.
uint32_t pair_grid(const Sched& sch, uint64_t tiles, uint32_t sms) {
    if (sch.dynamic) return static_cast<uint32_t>(std::max<uint64_t>(1, tiles));
    const uint32_t ctas = sch.num_ctas ? sch.num_ctas : sms;
    return static_cast<uint32_t>(std::min<uint64_t>(std::max(1u, ctas / 2), tiles));
}

// Operand of a GEMM as the kernel sees it: which index is contiguous, and
// whether TMA can fetch it (16-byte aligned base, pitch and batch stride).
struct OperandSpec {
    const void* ptr;
    uint32_t esize;
    uint64_t mn;          // rows of A (M) or columns of B (N) -- the MN extent
    uint64_t k;           // K
    int64_t ld;
    int64_t batch_stride;
    uint64_t batch;       // 1 for 2-D
    bool mn_major;
};

bool tma_ok(const OperandSpec& o) {
    const uintptr_t p = reinterpret_cast<uintptr_t>(o.ptr);
    if (p % 16) return false;
    if ((static_cast<uint64_t>(o.ld) * o.esize) % 16) return false;
    if (o.batch > 1 && (static_cast<uint64_t>(o.batch_stride) * o.esize) % 16) return false;
    if (o.batch > 1 && static_cast<uint64_t>(o.batch_stride) * o.esize >= (1ull << 40)) return false;
    if (static_cast<uint64_t>(o.ld) * o.esize >= (1ull << 40)) return false;
    return true;
}

uint32_t plain_vec(const OperandSpec& o) {
    uint32_t v = 16;
    const uint64_t p = reinterpret_cast<uintptr_t>(o.ptr);
    while (v > o.esize && (p % v || (static_cast<uint64_t>(o.ld) * o.esize) % v ||
                           (o.batch > 1 && (static_cast<uint64_t>(o.batch_stride) * o.esize) % v)))
        v >>= 1;
    return v;
}

bst_status encode(CUtensorMap* map, const OperandSpec& o, uint32_t tile_mn, CUtensorMapDataType dt) {
    if (!encoder()) return BST_ERR_CUDA;
    const uint32_t bk = kLine / o.esize;   // elements per 128-byte line
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    cuuint32_t estr[3] = {1, 1, 1};
    if (!o.mn_major) {
        dims[0] = o.k; dims[1] = o.mn;
        box[0] = bk; box[1] = tile_mn;
    } else {
        dims[0] = o.mn; dims[1] = o.k;
        box[0] = bk; box[1] = bk;
    }
    strides[0] = static_cast<cuuint64_t>(o.ld) * o.esize;
    uint32_t rank = 2;
    if (o.batch > 1 && o.batch_stride != 0) {
        dims[2] = o.batch;
        strides[1] = static_cast<cuuint64_t>(o.batch_stride) * o.esize;
        box[2] = 1;
        rank = 3;
    }
    CUresult r = g_encode(map, dt, rank, const_cast<void*>(o.ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BST_OK : BST_ERR_ALIGNMENT;
}

// An MN-major 16-bit operand whose row pitch is 8 bytes off a multiple of 16
// (ld = 4 mod 8 elements) has no tensor map, but pairs of its rows do: a
// view whose rows are two rows (ld + mn elements: row 2j whole, then the
// mn elements of row 2j+1; a pitch of 4*ld bytes) and whose K/2 rows end at
// the operand's last element.  Even rows are then boxes of 64 x 32 at x = n0,
// odd rows boxes of 72 x 32 at x = ld + n0 - 4, both 16-byte aligned.  Plain
// (unbatched) operands with an even K and a 16-byte-aligned base.
bool rows2_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("BST_ROWS2");
        return !(e && e[0] == '0');
    }();
    return on;
}

bool rows2_ok(const OperandSpec& o) {
    return o.mn_major && o.esize == 2 && o.batch == 1 && o.ld % 8 == 4 && o.k >= 2 && o.k % 2 == 0 &&
           reinterpret_cast<uintptr_t>(o.ptr) % 16 == 0 && static_cast<uint64_t>(o.ld) + o.mn < (1ull << 30);
}

bst_status encode_rows2(CUtensorMap* even, CUtensorMap* odd, const OperandSpec& o, CUtensorMapDataType dt) {
    if (!encoder()) return BST_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(o.ld) + o.mn, o.k / 2};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(o.ld) * 2 * o.esize};
    cuuint32_t estr[2] = {1, 1};
    cuuint32_t box_even[2] = {64, 32}, box_odd[2] = {72, 32};
    CUresult r = g_encode(even, dt, 2, const_cast<void*>(o.ptr), dims, strides, box_even, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return BST_ERR_ALIGNMENT;
    r = g_encode(odd, dt, 2, const_cast<void*>(o.ptr), dims, strides, box_odd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BST_OK : BST_ERR_ALIGNMENT;
}

bst_status fill_operand(OperandDesc& d, CUtensorMap* map, const OperandSpec& o, uint32_t tile_mn,
                        CUtensorMapDataType dt, bool require_tma) {
    d.ptr = static_cast<const uint8_t*>(o.ptr);
    d.ld = o.ld;
    d.batch_stride = o.batch_stride;
    d.mn_major = o.mn_major ? 1u : 0u;
    d.use_tma = tma_ok(o) ? 1u : 0u;
    d.vec_bytes = plain_vec(o);
    // a batch stride of 0 broadcasts one matrix to every batch: 2-D map, z ignored
    d.tma_rank = (o.batch > 1 && o.batch_stride != 0) ? 3u : 2u;
    d.rows2 = 0;
    if (!d.use_tma) {
        if (require_tma) return BST_ERR_ALIGNMENT;
        std::memset(map, 0, sizeof(*map));
        return BST_OK;
    }
    return encode(map, o, tile_mn, dt);
}


// fp16/bf16 tile choice among one-CTA 128 x {64,128,256} tiles and CTA-pair
// 256 x {128,256} tiles.  Cost = waves of tiles over the SMs (pairs count as
// one unit per two SMs) x per-tile time, the per-tile time being BN divided
// by how close that shape gets to the tensor peak when every SM pulls
// operands through L2 (narrow tiles need more operand bytes per flop).
struct TileChoice {
    uint32_t tm = kBM, bn = 128;
};

bst_status choose_tile(const Sched& sch, bool pair_ok, bool grouped, uint64_t M, uint64_t mult, uint64_t N,
                       uint32_t sms, TileChoice& out) {
    struct Cand {
        uint32_t tm, bn;
        double eff;
    };
    static const Cand cands[] = {{256, 256, 0.9}, {256, 128, 0.62}, {128, 256, 0.6}, {128, 128, 0.5}, {128, 64, 0.33}};
    if (sch.tile_m == 256 && !pair_ok) return BST_ERR_UNSUPPORTED;
    double best = 1e300;
    for (const Cand& c : cands) {
        if ((sch.tile_m && c.tm != sch.tile_m) || (sch.tile_n && c.bn != sch.tile_n)) continue;
        if (c.tm == 256 && !pair_ok) continue;
        const uint64_t lm = grouped ? (M + c.tm - 1) / c.tm + mult : ((M + c.tm - 1) / c.tm) * mult;
        const uint64_t tiles = lm * ((N + c.bn - 1) / c.bn);
        const uint64_t units = c.tm == 256 ? std::max(1u, sms / 2) : sms;
        const double cost = static_cast<double>((tiles + units - 1) / units) * c.bn / c.eff;
        if (cost < best * 0.999) {
            best = cost;
            out.tm = c.tm;
            out.bn = c.bn;
        }
    }
    return best < 1e300 ? BST_OK : BST_ERR_UNSUPPORTED;
}

// Small problems are bound by the DRAM latency of their first touches: when
// the operands' storage fits well inside L2 the kernel prefetches all of it
// at start.  BST_PREFETCH_MB sets the limit (0 disables).
void set_prefetch(GemmArgs& g, const OperandSpec& a, const OperandSpec& b, const uint8_t* s1, uint64_t s1_bytes,
                  const uint8_t* s2, uint64_t s2_bytes) {
    static const uint64_t limit = [] {
        const char* e = std::getenv("BST_PREFETCH_MB");
        return (e ? std::strtoull(e, nullptr, 10) : 32ull) << 20;
    }();
    auto span = [](const OperandSpec& o) {
        const uint64_t rows = o.mn_major ? o.k : o.mn;          // rows of storage
        const uint64_t per = static_cast<uint64_t>(o.ld) * (rows ? rows - 1 : 0) + (o.mn_major ? o.mn : o.k);
        const uint64_t slab = per * o.esize;
        return o.batch > 1 ? static_cast<uint64_t>(o.batch_stride) * o.esize * (o.batch - 1) + slab : slab;
    };
    const uint64_t ab = span(a), bb = span(b);
    for (int i = 0; i < 4; ++i) { g.pf_ptr[i] = nullptr; g.pf_bytes[i] = 0; }
    if (ab + bb + s1_bytes + s2_bytes > limit) return;
    g.pf_ptr[0] = static_cast<const uint8_t*>(a.ptr); g.pf_bytes[0] = ab;
    g.pf_ptr[1] = static_cast<const uint8_t*>(b.ptr); g.pf_bytes[1] = bb;
    g.pf_ptr[2] = s1; g.pf_bytes[2] = s1 ? s1_bytes : 0;
    g.pf_ptr[3] = s2; g.pf_bytes[3] = s2 ? s2_bytes : 0;
}

// Widest store (16, 8, 4 or 2 bytes, at least the element size) that every
// row start of an output allows: the base address, the row pitch and the
// batch stride in bytes must all be multiples of it.
uint32_t store_vec(const void* ptr, int64_t ld_bytes, int64_t batch_stride_bytes, uint32_t esize) {
    uint32_t v = 16;
    const uint64_t p = reinterpret_cast<uintptr_t>(ptr);
    while (v > esize && (p % v || static_cast<uint64_t>(ld_bytes) % v || static_cast<uint64_t>(batch_stride_bytes) % v))
        v >>= 1;
    return v;
}

// Split-K on CTA-pair tiles (256 x 256 or 256 x 128) for problems whose
// tiles cannot fill the GPU.  Among the shapes whose clusters of 2*S CTAs
// (one per tile) all fit on the SMs and are resident at once, with at least
// 4 k-blocks per split, it takes the one with the fewest k-block time units
// per cluster: a 256 x 128 k-block costs about 0.6 of a 256 x 256 one (it is
// shared-memory-port bound, the wide one tensor bound).  splits = 1: no
// split; splits = 0: the caller forced a split this problem cannot take.
struct SplitChoice {
    uint32_t splits = 1;
    uint32_t bn = 256;
};

SplitChoice choose_splits(const Sched& sch, bool eligible, uint64_t M, uint64_t N, uint32_t num_kb, uint32_t sms) {
    SplitChoice none;
    if (sch.split_k == 1 || sch.dynamic) return none;
    const bool forced = sch.split_k >= 2;
    const bool bn_ok = sch.tile_n == 0 || sch.tile_n == 128 || sch.tile_n == 256;
    if (!eligible || (sch.tile_m && sch.tile_m != 256) || !bn_ok) {
        if (forced) none.splits = 0;
        return none;
    }
    auto tiles_of = [&](uint64_t bn) { return ((M + 255) / 256) * ((N + bn - 1) / bn); };
    if (forced) {
        SplitChoice c;
        c.splits = sch.split_k;
        c.bn = sch.tile_n ? sch.tile_n : 256;
        return c;
    }
    if (tiles_of(256) * 2 * 2 > sms) return none;     // pairs alone already fill half the GPU or more
    SplitChoice best;
    double best_cost = 0;
    for (uint32_t bn : {256u, 128u}) {
        if (sch.tile_n && sch.tile_n != bn) continue;
        const uint64_t tiles = tiles_of(bn);
        for (uint32_t s : {4u, 2u}) {
            uint32_t resident = 0;
            if (tiles * 2 * s > sms || num_kb < 4 * s) continue;
            if (splitk_resident_clusters(bn, s, &resident) != cudaSuccess) { cudaGetLastError(); continue; }
            if (tiles > resident) continue;
            const double cost = static_cast<double>((num_kb + s - 1) / s) * (bn == 256 ? 1.0 : 0.6);
            if (best.splits == 1 || cost < best_cost) {
                best.splits = s;
                best.bn = bn;
                best_cost = cost;
            }
        }
    }
    return best;
}

// Split-K of one-CTA tiles for fp16/bf16 operands that TMA cannot fetch.
// Their copies go through the load/store units, whose issue rate per SM is
// the limit (about 0.6 us per 8 KB k-block of copied operand): when the tiles
// leave SMs idle, spreading each tile's k-blocks over a cluster of S CTAs
// divides the copy time per CTA, for the exchange of the partials through
// distributed shared memory (about 1 us per 32 KB received).  Cost, in units
// of one 8 KB copy: k-blocks per CTA x copied KB per k-block / 8, plus the
// exchange; the split is taken when it beats the unsplit tile.  splits = 0:
// a forced split this problem cannot take.
SplitChoice choose_copy_splits(const Sched& sch, bool eligible, bool a_copied, bool b_copied, uint64_t M,
                               uint64_t N, uint32_t num_kb, uint32_t sms, uint32_t bn_unsplit) {
    SplitChoice none;
    if (sch.split_k == 1 || sch.dynamic) return none;
    const bool forced = sch.split_k >= 2;
    if (!eligible || (sch.tile_m && sch.tile_m != 128)) {
        if (forced) none.splits = 0;
        return none;
    }
    auto copy_units = [&](uint32_t bn) { return ((a_copied ? 16.0 : 0.0) + (b_copied ? bn * 0.125 : 0.0)) / 8.0; };
    auto tiles_of = [&](uint64_t bn) { return ((M + 127) / 128) * ((N + bn - 1) / bn); };
    const uint64_t t1 = tiles_of(bn_unsplit);
    double best_cost = static_cast<double>((t1 + sms - 1) / sms) * num_kb * copy_units(bn_unsplit);
    SplitChoice best;
    const std::pair<uint32_t, uint32_t> cands[] = {{64u, 2u}, {128u, 2u}, {128u, 4u}};
    for (const auto& c : cands) {
        const uint32_t bn = c.first, s = c.second;
        if (sch.tile_n && sch.tile_n != bn) continue;
        if (forced && sch.split_k != s) continue;
        const uint64_t tiles = tiles_of(bn);
        uint32_t resident = 0;
        if (!forced && (tiles * s > sms || num_kb < s)) continue;
        if (dense_split_resident(bn, s, &resident) != cudaSuccess) { cudaGetLastError(); continue; }
        if (resident == 0 || (!forced && tiles > resident)) continue;
        const double xchg = (s - 1) * (128.0 * bn / s * 4.0) / 32768.0 * (1.0 / 0.6);
        const double cost = ((num_kb + s - 1) / s) * copy_units(bn) + xchg;
        if (forced ? (best.splits == 1) : cost < best_cost * 0.95) {
            best.splits = s;
            best.bn = bn;
            best_cost = cost;
        }
    }
    if (forced && best.splits == 1) best.splits = 0;
    return best;
}

CUtensorMapDataType tmap_type(bst_dtype t) {
    if (t == BST_F16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (t == BST_BF16) return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return CU_TENSOR_MAP_DATA_TYPE_UINT8;
}

bst_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BST_OK : BST_ERR_CUDA; }

constexpr uint64_t kMaxDim = (1ull << 31) - 1;

// A [M,K] / B [K,N] logical -> operand specs.  Row-major A is K-contiguous;
// row-major B is N-contiguous (MN-major).
bst_status make_specs(uint64_t M, uint64_t N, uint64_t K, const void* A, bst_layout la, int64_t lda, int64_t sa,
                      const void* B, bst_layout lb, int64_t ldb, int64_t sb, uint32_t esize, uint64_t batch,
                      OperandSpec& a, OperandSpec& b) {
    if (la != BST_ROW_MAJOR && la != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    if (lb != BST_ROW_MAJOR && lb != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    a = OperandSpec{A, esize, M, K, lda, sa, batch, la == BST_COL_MAJOR};
    b = OperandSpec{B, esize, N, K, ldb, sb, batch, lb == BST_ROW_MAJOR};
    const uint64_t a_contig = a.mn_major ? M : K;
    const uint64_t b_contig = b.mn_major ? N : K;
    if (lda < 1 || static_cast<uint64_t>(lda) < a_contig) return BST_ERR_INVALID_ARG;
    if (ldb < 1 || static_cast<uint64_t>(ldb) < b_contig) return BST_ERR_INVALID_ARG;
    return BST_OK;
}

bst_status run_dense(uint32_t mode, int64_t M, int64_t N, int64_t K, const void* A, bst_dtype at, bst_layout la,
                     int64_t lda, int64_t sa, const void* B, bst_dtype bt, bst_layout lb, int64_t ldb, int64_t sb,
                     void* C, bst_dtype ct, int64_t ldc, int64_t sc, int64_t batch, const bst_sched* sched_in,
                     void* stream_v) {
    if (M < 0 || N < 0 || K < 0 || batch < 1) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(M) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(K) > kMaxDim || static_cast<uint64_t>(batch) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (at != bt || (at != BST_F16 && at != BST_BF16)) return BST_ERR_UNSUPPORTED;
    uint32_t c_code;
    if (!out_code(ct, c_code)) return BST_ERR_UNSUPPORTED;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (mode == kModeBatched && (sa < 0 || sb < 0 || sc < 0)) return BST_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BST_OK;
    if (!C || (K > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    OperandSpec a, b;
    if (bst_status s = make_specs(M, N, K, A, la, lda, sa, B, lb, ldb, sb, 2, static_cast<uint64_t>(batch), a, b))
        return s;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const uint32_t csize = dtype_bytes(ct);
    if (K == 0)
        return cuda_status(launch_zero_fill(static_cast<uint8_t*>(C), ldc, sc, M, N, batch, csize, dev.sms, stream));

    const bool pair_ok = tma_ok(a) && tma_ok(b);
    const uint32_t num_kb = static_cast<uint32_t>((K + 63) / 64);
    SplitChoice sc_k = choose_splits(sch, pair_ok && mode == kModePlain, M, N, num_kb, dev.sms);
    TileChoice tc;
    bool copy_split = false;
    // B through the two-row view (one-CTA 128 x 64 tiles, no split)
    const bool b_rows2 = !pair_ok && mode == kModePlain && tma_ok(a) && rows2_ok(b) && rows2_enabled() &&
                         (sch.tile_m == 0 || sch.tile_m == 128) && (sch.tile_n == 0 || sch.tile_n == 64) &&
                         sch.split_k <= 1;
    if (b_rows2) {
        tc.tm = 128;
        tc.bn = 64;
    } else if (!pair_ok) {
        // operands TMA cannot fetch: one-CTA tiles, optionally split along K
        Sched plain = sch;
        plain.split_k = 0;
        if (bst_status s = choose_tile(plain, false, false, M, batch, N, dev.sms, tc)) return s;
        sc_k = choose_copy_splits(sch, mode == kModePlain, !tma_ok(a), !tma_ok(b), M, N, num_kb, dev.sms, tc.bn);
        copy_split = sc_k.splits > 1;
        if (copy_split) tc.bn = sc_k.bn;
    }
    const uint32_t splits = sc_k.splits;
    if (splits == 0) return BST_ERR_UNSUPPORTED;
    if (splits > 1 && !copy_split) { tc.tm = 256; tc.bn = sc_k.bn; }
    else if (pair_ok) {
        if (bst_status s = choose_tile(sch, pair_ok, false, M, batch, N, dev.sms, tc)) return s;
    }
    const uint32_t bn = tc.bn;
    const bool pair = tc.tm == 256;
    const uint64_t tiles = ((M + tc.tm - 1) / tc.tm) * ((N + bn - 1) / bn) * batch;
    if (tiles >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    const uint32_t smem_need = b_rows2 ? smem_dense_rows2()
                               : copy_split ? smem_dense_split(bn, splits)
                               : splits > 1 ? smem_splitk(bn, splits) : pair ? smem_pair(bn, 0) : smem_dense(bn, 0);
    if (smem_need == 0 || smem_need > dev.max_smem) return BST_ERR_UNSUPPORTED;

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, a, kBM, tmap_type(at), false)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, b, pair ? bn / 2 : bn, tmap_type(bt), false)) return s;
    if (b_rows2) {
        if (bst_status s = encode_rows2(&p.tmap_sfa, &p.tmap_sfb, b, tmap_type(bt))) return s;
        p.g.b.rows2 = 1;
    }
    p.g.M = M; p.g.N = N; p.g.K = K;
    p.g.batch = batch;
    p.g.mode = mode;
    p.g.ab_fmt = at == BST_BF16 ? 1u : 0u;
    p.g.esize = 2;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.ps.init(static_cast<uint32_t>(M), static_cast<uint32_t>(N), tc.tm, bn, sch.offset, sch.dir);
    p.g.num_kb = (K + 63) / 64;
    p.g.chunk_kb = p.g.num_kb;
    p.g.total_tiles = static_cast<uint32_t>(tiles);
    p.g.C = static_cast<uint8_t*>(C);
    p.g.ldc = ldc;
    p.g.c_batch_stride = sc;
    p.g.c_type = c_code;
    p.g.c_vec = store_vec(C, ldc * csize, mode == kModeBatched ? sc * csize : 0, csize);
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    set_prefetch(p.g, a, b, nullptr, 0, nullptr, 0);
    const uint32_t ctas = sch.num_ctas ? sch.num_ctas : dev.sms;
    if (copy_split) return cuda_status(launch_dense_split(p, bn, splits, static_cast<uint32_t>(tiles), stream));
    if (splits > 1) return cuda_status(launch_pair_splitk(p, bn, splits, static_cast<uint32_t>(tiles), stream));
    if (pair)
        return cuda_status(launch_pair(p, bn, pair_grid(sch, tiles, dev.sms),
                                       stream));
    const uint32_t grid = static_cast<uint32_t>(std::min<uint64_t>(ctas, tiles));
    return cuda_status(launch_dense(p, bn, grid, stream));
}

// MXFP8 tile shape and split-K.  One-CTA 128 x {128, 256} tiles cost about
// 0.41 / 0.44 us per k-block (the MMA loop with the operands arriving from
// DRAM; it barely depends on the width), so wide tiles win whenever they can
// fill the GPU; split-K over clusters of S CTAs (one tile per cluster) lets
// 128 x 256 tiles do so, at about 4 us for the cluster launch and the
// exchange and finish of the partials through distributed shared memory.
// CTA-pair 256 x {128, 256} tiles (operands and scale-factor arrays that TMA
// can address, K a multiple of 1024) need no exchange: about 0.27 / 0.31 us
// per k-block per pair (measured on 1024 x 2048 x 4096), two SMs per tile.
// Cost = waves x k-blocks per CTA x per-k-block time (+ the split cost).
// splits = 0 on return: a forced split this problem cannot take.
bst_status choose_mx(const Sched& sch, uint64_t M, uint64_t N, uint32_t num_kb, uint32_t sms, bool pair_ok,
                     uint32_t& tm, uint32_t& bn, uint32_t& splits) {
    const uint64_t loops_m = (M + kBM - 1) / kBM;
    auto tiles_of = [&](uint32_t w) { return loops_m * ((N + w - 1) / w); };
    auto split_ok = [&](uint32_t w, uint32_t s) {
        uint32_t resident = 0;
        if (mxf8_split_resident(w, s, &resident) != cudaSuccess) { cudaGetLastError(); return false; }
        return resident > 0 && tiles_of(w) <= resident && tiles_of(w) * s <= sms;
    };
    if (sch.tile_m == 256 && (!pair_ok || sch.split_k >= 2)) return BST_ERR_UNSUPPORTED;
    if (sch.split_k >= 2) {
        tm = kBM;
        bn = sch.tile_n ? sch.tile_n : (sch.split_k == 2 ? 256u : 128u);
        splits = sch.split_k;
        uint32_t resident = 0;
        if (mxf8_split_resident(bn, splits, &resident) != cudaSuccess || resident == 0) {
            cudaGetLastError();
            return BST_ERR_UNSUPPORTED;
        }
        return BST_OK;
    }
    double best = 1e300;
    bn = 0;
    if (sch.tile_m != 256) {
        for (uint32_t w : {128u, 256u}) {
            if (sch.tile_n && sch.tile_n != w) continue;
            for (uint32_t s : {1u, 2u, 4u}) {
                if (s > 1 && (sch.split_k == 1 || num_kb < 4 * s || !split_ok(w, s))) continue;
                const uint64_t ctas = s > 1 ? tiles_of(w) * s : tiles_of(w);
                const double waves = static_cast<double>((ctas + sms - 1) / sms);
                const double cost = waves * ((num_kb + s - 1) / s) * (w == 256 ? 0.44 : 0.41) + (s > 1 ? 4.0 : 0.0);
                if (cost < best * 0.999) { best = cost; tm = kBM; bn = w; splits = s; }
            }
        }
    }
    if (pair_ok && sch.tile_m != kBM) {
        for (uint32_t w : {128u, 256u}) {
            if (sch.tile_n && sch.tile_n != w) continue;
            const uint64_t tiles = ((M + 255) / 256) * ((N + w - 1) / w);
            const uint64_t units = std::max(1u, sms / 2);
            const double waves = static_cast<double>((tiles + units - 1) / units);
            const double cost = waves * num_kb * (w == 256 ? 0.31 : 0.27);
            if (cost < best * 0.999) { best = cost; tm = 256; bn = w; splits = 1; }
        }
    }
    return bn ? BST_OK : BST_ERR_UNSUPPORTED;
}

bst_status run_mxf8(int64_t M, int64_t N, int64_t K, const void* A, bst_layout la, int64_t lda, const void* B,
                    bst_layout lb, int64_t ldb, void* C, bst_dtype ct, int64_t ldc, const uint8_t* sfa,
                    const uint8_t* sfb, const bst_sched* sched_in, void* stream_v) {
    if (M < 0 || N < 0 || K < 0) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(M) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(K) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    uint32_t c_code;
    if (!out_code(ct, c_code)) return BST_ERR_UNSUPPORTED;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if (sch.dynamic || sch.shuffle_k) return BST_ERR_UNSUPPORTED;   // one-CTA MXFP8 tiles, fixed K order
    if (la != BST_ROW_MAJOR || lb != BST_COL_MAJOR) return BST_ERR_UNSUPPORTED;
    if (K % 128) return BST_ERR_UNSUPPORTED;
    if (sch.tile_n == 64 || (sch.tile_m && sch.tile_m != kBM && sch.tile_m != 256)) return BST_ERR_UNSUPPORTED;
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BST_OK;
    if (!C || (K > 0 && (!A || !B || !sfa || !sfb))) return BST_ERR_INVALID_ARG;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(sfa) | reinterpret_cast<uintptr_t>(sfb)) % 4))
        return BST_ERR_ALIGNMENT;
    OperandSpec a, b;
    if (bst_status s = make_specs(M, N, K, A, la, lda, 0, B, lb, ldb, 0, 1, 1, a, b)) return s;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const uint32_t csize = dtype_bytes(ct);
    if (K == 0) return cuda_status(launch_zero_fill(static_cast<uint8_t*>(C), ldc, 0, M, N, 1, csize, dev.sms, stream));
    const uint32_t num_kb = static_cast<uint32_t>(K / 128);
    // scale factors by TMA when each row's codes are a whole number of 16-byte
    // groups (K a multiple of 512) and both arrays start 16-byte aligned;
    // otherwise the scale warp copies them row by row (one-CTA tiles only)
    const bool sf_tma = K % 512 == 0 && reinterpret_cast<uintptr_t>(sfa) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(sfb) % 16 == 0;
    uint32_t tm = kBM, bn = 0, splits = 1;
    // CTA pairs take the codes in groups of 8 k-blocks (K a multiple of 1024)
    const bool pair_ok = sf_tma && K % 1024 == 0 && tma_ok(a) && tma_ok(b);
    if (bst_status s = choose_mx(sch, M, N, num_kb, dev.sms, pair_ok, tm, bn, splits))
        return s;
    const bool pair = tm == 256;
    const uint64_t tiles = ((M + tm - 1) / tm) * ((N + bn - 1) / bn);
    if (tiles >= (1ull << 31)) return BST_ERR_INVALID_ARG;
    if ((pair ? smem_mxf8_pair(bn) : smem_mxf8(bn)) > dev.max_smem) return BST_ERR_UNSUPPORTED;

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, a, kBM, CU_TENSOR_MAP_DATA_TYPE_UINT8, true)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, b, pair ? bn / 2 : bn, CU_TENSOR_MAP_DATA_TYPE_UINT8, true))
        return s;
    p.g.M = M; p.g.N = N; p.g.K = K;
    p.g.batch = 1;
    p.g.mode = kModePlain;
    p.g.esize = 1;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.ps.init(static_cast<uint32_t>(M), static_cast<uint32_t>(N), tm, bn, sch.offset, sch.dir);
    p.g.num_kb = K / 128;
    p.g.chunk_kb = p.g.num_kb;
    p.g.total_tiles = static_cast<uint32_t>(tiles);
    p.g.C = static_cast<uint8_t*>(C);
    p.g.ldc = ldc;
    p.g.c_type = c_code;
    p.g.c_vec = store_vec(C, ldc * csize, 0, csize);
    p.g.sfa = sfa;
    p.g.sfb = sfb;
    p.g.sf_ld = static_cast<uint32_t>(K / 32);
    if (sf_tma) {
        if (!encoder()) return BST_ERR_CUDA;
        const cuuint64_t row_bytes = static_cast<cuuint64_t>(K / 32);
        cuuint32_t estr[2] = {1, 1};
        cuuint64_t dims_a[2] = {row_bytes, static_cast<cuuint64_t>(M)};
        cuuint64_t dims_b[2] = {row_bytes, static_cast<cuuint64_t>(N)};
        cuuint64_t strides[1] = {row_bytes};
        // one-CTA tiles take 16 bytes (4 k-blocks) of codes per row per load,
        // CTA pairs 32 (8 k-blocks), all of a tile's B columns in each CTA
        const cuuint32_t row_box = pair ? 32 : 16;
        cuuint32_t box_a[2] = {row_box, kBM};
        cuuint32_t box_b[2] = {row_box, bn};
        if (g_encode(&p.tmap_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(sfa), dims_a, strides, box_a,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            g_encode(&p.tmap_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(sfb), dims_b, strides, box_b,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return BST_ERR_CUDA;
        p.g.sf_tma = 1;
    }
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    set_prefetch(p.g, a, b, sfa, static_cast<uint64_t>(M) * (K / 32), sfb, static_cast<uint64_t>(N) * (K / 32));
    if (splits > 1) return cuda_status(launch_mxf8_split(p, bn, splits, static_cast<uint32_t>(tiles), stream));
    if (pair) return cuda_status(launch_mxf8_pair(p, bn, pair_grid(sch, tiles, dev.sms), stream));
    const uint32_t ctas = sch.num_ctas ? sch.num_ctas : dev.sms;
    const uint32_t grid = static_cast<uint32_t>(std::min<uint64_t>(ctas, tiles));
    return cuda_status(launch_mxf8(p, bn, grid, stream));
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }


}  // namespace
}  // namespace bst

using namespace bst;

namespace {

// Shared by the bf16 and the int8 slice-K entry points once the operands are
// 16-bit and TMA-addressable: builds the whole-operand maps, launches the
// per-group set-up and then the CTA-pair GEMM in slice-K mode.
struct SliceKRun {
    OperandSpec a, b;      // A: MN extent M, K total_k; B: MN extent N
    uint32_t ab_fmt;       // kind::f16 format: 0 f16, 1 bf16
    CUtensorMapDataType dt;
    uint32_t c_code, csize;
    void* C;
    int64_t ldc, stride_c;
    const float* scale_a = nullptr;
    const float* scale_b = nullptr;
    int64_t stride_sa = 0, stride_sb = 0;
    int32_t* acc_out = nullptr;
    bool dequant = false;
};

bst_status run_slice_k(const SliceKRun& r, int32_t G, const int32_t* group_k, int64_t M, int64_t N,
                       int64_t total_k, uint8_t* meta, const Sched& sch, const DeviceInfo& dev, cudaStream_t stream) {
    uint32_t bn = 256;
    if (r.dequant) {
        if (sch.tile_n != 0 && sch.tile_n != 256) return BST_ERR_UNSUPPORTED;
    } else {
        Sched pair_only = sch;
        pair_only.tile_m = 256;
        TileChoice tc;
        if (bst_status s = choose_tile(pair_only, true, false, M, G, N, dev.sms, tc)) return s;
        bn = tc.bn;
    }
    const uint64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn) * static_cast<uint64_t>(G);
    if (tiles >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    const uint32_t smem_need = r.dequant ? smem_pair_dequant() + 8 * (static_cast<uint32_t>(G) + 1)
                                         : smem_pair(bn, static_cast<uint32_t>(G));
    if (smem_need > dev.max_smem) return BST_ERR_UNSUPPORTED;
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, r.a, kBM, r.dt, true)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, r.b, bn / 2, r.dt, true)) return s;
    uint8_t* maps = meta;
    uint32_t* group_kb = reinterpret_cast<uint32_t*>(meta + static_cast<size_t>(G) * 256);
    // bytes between consecutive K indices, and which map dimension runs along K
    const uint64_t a_kstep = r.a.mn_major ? static_cast<uint64_t>(r.a.ld) * r.a.esize : r.a.esize;
    const uint64_t b_kstep = r.b.mn_major ? static_cast<uint64_t>(r.b.ld) * r.b.esize : r.b.esize;
    cudaError_t e = launch_slice_k_prep(p.tmap_a, p.tmap_b, group_k, static_cast<uint32_t>(G),
                                        static_cast<uint64_t>(total_k), r.a.ptr, a_kstep, r.a.mn_major ? 1u : 0u,
                                        r.b.ptr, b_kstep, r.b.mn_major ? 1u : 0u, maps, group_kb, dev.err, stream);
    if (e != cudaSuccess) return BST_ERR_CUDA;
    p.g.M = M; p.g.N = N; p.g.K = total_k;
    p.g.batch = static_cast<uint32_t>(G);
    p.g.mode = kModeSliceK;
    p.g.ab_fmt = r.ab_fmt;
    p.g.esize = 2;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.ps.init(static_cast<uint32_t>(M), static_cast<uint32_t>(N), 256, bn, sch.offset, sch.dir);
    p.g.num_kb = (total_k + 63) / 64;
    p.g.chunk_kb = r.dequant ? kDequantChunkK / 64 : p.g.num_kb;
    p.g.total_tiles = static_cast<uint32_t>(tiles);
    p.g.G = static_cast<uint32_t>(G);
    p.g.kmaps = maps;
    p.g.group_kb = group_kb;
    p.g.C = static_cast<uint8_t*>(r.C);
    p.g.ldc = r.ldc;
    p.g.c_batch_stride = r.stride_c;
    p.g.c_type = r.c_code;
    p.g.c_vec = store_vec(r.C, r.ldc * r.csize, r.stride_c * r.csize, r.csize);
    p.g.scale_a = r.scale_a;
    p.g.scale_b = r.scale_b;
    p.g.sa_group_stride = r.stride_sa;
    p.g.sb_group_stride = r.stride_sb;
    p.g.acc_out = r.acc_out;
    p.g.acc_vec = r.acc_out ? store_vec(r.acc_out, r.ldc * 4, r.stride_c * 4, 4) : 4u;
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    const uint32_t pairs = pair_grid(sch, tiles, dev.sms);
    return cuda_status(r.dequant ? launch_pair_dequant(p, pairs, stream) : launch_pair(p, bn, pairs, stream));
}

}  // namespace

extern "C" {

bst_status bst_gemm(int64_t M, int64_t N, int64_t K, const void* A, bst_dtype a_type, bst_layout a_layout,
                    int64_t lda, const void* B, bst_dtype b_type, bst_layout b_layout, int64_t ldb, void* C,
                    bst_dtype c_type, int64_t ldc, const uint8_t* scale_a, const uint8_t* scale_b,
                    const bst_sched* sched, void* stream) {
    if (a_type == BST_E4M3 || b_type == BST_E4M3) {
        if (a_type != b_type) return BST_ERR_UNSUPPORTED;
        return run_mxf8(M, N, K, A, a_layout, lda, B, b_layout, ldb, C, c_type, ldc, scale_a, scale_b, sched, stream);
    }
    if (scale_a || scale_b) return BST_ERR_INVALID_ARG;
    return run_dense(kModePlain, M, N, K, A, a_type, a_layout, lda, 0, B, b_type, b_layout, ldb, 0, C, c_type, ldc,
                     0, 1, sched, stream);
}

bst_status bst_gemm_batched(int64_t M, int64_t N, int64_t K, const void* A, bst_dtype a_type, bst_layout a_layout,
                            int64_t lda, int64_t stride_a, const void* B, bst_dtype b_type, bst_layout b_layout,
                            int64_t ldb, int64_t stride_b, void* C, bst_dtype c_type, int64_t ldc, int64_t stride_c,
                            int64_t batch, const bst_sched* sched, void* stream) {
    return run_dense(batch > 1 ? kModeBatched : kModePlain, M, N, K, A, a_type, a_layout, lda, stride_a, B, b_type,
                     b_layout, ldb, stride_b, C, c_type, ldc, stride_c, batch, sched, stream);
}

bst_status bst_gemm_grouped(int32_t G, const int32_t* group_m, int64_t total_m, int64_t N, int64_t K, const void* A,
                            int64_t lda, const void* B, bst_layout b_layout, int64_t ldb, int64_t stride_b, void* C,
                            int64_t ldc, bst_dtype ab_type, bst_dtype c_type, const bst_sched* sched_in,
                            void* stream_v) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || total_m < 0 || N < 0 || K < 0 || stride_b < 0)
        return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(total_m) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(K) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (ab_type != BST_F16 && ab_type != BST_BF16) return BST_ERR_UNSUPPORTED;
    uint32_t c_code;
    if (!out_code(c_type, c_code)) return BST_ERR_UNSUPPORTED;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (total_m == 0 || N == 0) return BST_OK;
    if (!group_m || !C || (K > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    OperandSpec a, b;
    if (bst_status s = make_specs(total_m, N, K, A, BST_ROW_MAJOR, lda, 0, B, b_layout, ldb, stride_b, 2, 1, a, b))
        return s;
    b.batch = static_cast<uint64_t>(G);
    if (G > 1 && stride_b < 1) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const uint32_t csize = dtype_bytes(c_type);
    if (K == 0)
        return cuda_status(
            launch_zero_fill(static_cast<uint8_t*>(C), ldc, 0, total_m, N, 1, csize, dev.sms, stream));
    TileChoice tc;
    if (bst_status s = choose_tile(sch, tma_ok(a) && tma_ok(b), true, total_m, G, N, dev.sms, tc)) return s;
    const uint32_t bn = tc.bn;
    const bool pair = tc.tm == 256;
    // an upper bound of the tile count: sum ceil(M_g/tm) <= total_m/tm + G
    const uint64_t loops_m_bound = (total_m + tc.tm - 1) / tc.tm + G;
    const uint64_t tiles_bound = loops_m_bound * ((N + bn - 1) / bn);
    if (tiles_bound >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    if ((pair ? smem_pair(bn, G) : smem_dense(bn, G)) > dev.max_smem) return BST_ERR_UNSUPPORTED;

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, a, kBM, tmap_type(ab_type), false)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, b, pair ? bn / 2 : bn, tmap_type(ab_type), false)) return s;
    p.g.M = 0; p.g.N = N; p.g.K = K;
    p.g.batch = 1;
    p.g.mode = kModeGrouped;
    p.g.ab_fmt = ab_type == BST_BF16 ? 1u : 0u;
    p.g.esize = 2;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.num_kb = (K + 63) / 64;
    p.g.chunk_kb = p.g.num_kb;
    p.g.group_m = group_m;
    p.g.G = static_cast<uint32_t>(G);
    p.g.total_m = static_cast<uint32_t>(total_m);
    p.g.C = static_cast<uint8_t*>(C);
    p.g.ldc = ldc;
    p.g.c_type = c_code;
    p.g.c_vec = store_vec(C, ldc * csize, 0, csize);
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles_bound);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    set_prefetch(p.g, a, b, nullptr, 0, nullptr, 0);
    const uint32_t ctas = sch.num_ctas ? sch.num_ctas : dev.sms;
    if (pair)
        return cuda_status(launch_pair(
            p, bn, pair_grid(sch, tiles_bound, dev.sms), stream));
    const uint32_t grid = static_cast<uint32_t>(std::min<uint64_t>(ctas, tiles_bound));
    return cuda_status(launch_dense(p, bn, grid, stream));
}

size_t bst_gemm_quant_per_token_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    const size_t kp = static_cast<size_t>((K + 7) / 8 * 8);
    const size_t np = static_cast<size_t>((N + 7) / 8 * 8);
    const size_t a = static_cast<size_t>(M) * kp * 2;
    const size_t b = std::max(static_cast<size_t>(N) * kp, static_cast<size_t>(K) * np) * 2;
    return round256(a) + round256(b);
}

bst_status bst_gemm_quant_per_token(int64_t M, int64_t N, int64_t K, const int8_t* A, int64_t lda, const int8_t* B,
                                    bst_layout b_layout, int64_t ldb, const float* scale_a, const float* scale_b,
                                    void* C, int64_t ldc, int32_t* acc_out, void* workspace, size_t workspace_bytes,
                                    const bst_sched* sched_in, void* stream_v) {
    if (M < 0 || N < 0 || K < 0) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(M) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(K) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (b_layout != BST_ROW_MAJOR && b_layout != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    // tiles: 256 x 256 CTA pairs (the default) or 128 x 128 single CTAs
    if (sch.tile_m != 0 && sch.tile_m != 128 && sch.tile_m != 256) return BST_ERR_UNSUPPORTED;
    if (sch.tile_n != 0 && sch.tile_n != 128 && sch.tile_n != 256) return BST_ERR_UNSUPPORTED;
    if ((sch.tile_m == 256 && sch.tile_n == 128) || (sch.tile_m == 128 && sch.tile_n == 256)) return BST_ERR_UNSUPPORTED;
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (lda < 1 || lda < K) return BST_ERR_INVALID_ARG;
    if (ldb < 1 || ldb < (b_layout == BST_COL_MAJOR ? K : N)) return BST_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BST_OK;
    if (!C || !scale_a || !scale_b || (K > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (K == 0) {
        cudaError_t e = launch_zero_fill(static_cast<uint8_t*>(C), ldc, 0, M, N, 1, 2, dev.sms, stream);
        if (e == cudaSuccess && acc_out)
            e = launch_zero_fill(reinterpret_cast<uint8_t*>(acc_out), ldc, 0, M, N, 1, 4, dev.sms, stream);
        return cuda_status(e);
    }
    const size_t need = bst_gemm_quant_per_token_workspace_size(M, N, K);
    if (!workspace || workspace_bytes < need) return BST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return BST_ERR_ALIGNMENT;
    const int64_t kp = (K + 7) / 8 * 8;
    const int64_t np = (N + 7) / 8 * 8;
    uint16_t* wa = static_cast<uint16_t*>(workspace);
    uint16_t* wb = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + round256(static_cast<size_t>(M) * kp * 2));
    const bool b_kmajor = b_layout == BST_COL_MAJOR;   // stored [N, K]
    const int64_t ldwb = b_kmajor ? kp : np;
    const bool pair = sch.tile_m == 256 || sch.tile_n == 256 ||
                      (sch.tile_m == 0 && sch.tile_n == 0 && M > kBM && N > 128);
    const uint32_t tm = pair ? 2 * kBM : kBM, tn = pair ? 256u : 128u;
    const uint64_t tiles = ((M + tm - 1) / tm) * ((N + tn - 1) / tn);
    if (tiles >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    if ((pair ? smem_pair_dequant() : smem_dequant()) > dev.max_smem) return BST_ERR_UNSUPPORTED;

    const WidenArgs wa_args{A, lda, wa, kp, M, K};
    const WidenArgs wb_args = b_kmajor ? WidenArgs{B, ldb, wb, ldwb, N, K} : WidenArgs{B, ldb, wb, ldwb, K, N};
    if (launch_widen2_s8_bf16(wa_args, wb_args, dev.sms, stream, dev.err, timeout_ns()) != cudaSuccess)
        return BST_ERR_CUDA;

    OperandSpec a{wa, 2, static_cast<uint64_t>(M), static_cast<uint64_t>(K), kp, 0, 1, false};
    OperandSpec b{wb, 2, static_cast<uint64_t>(N), static_cast<uint64_t>(K), ldwb, 0, 1, !b_kmajor};
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, a, kBM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, true)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, b, 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, true)) return s;
    p.g.M = M; p.g.N = N; p.g.K = K;
    p.g.batch = 1;
    p.g.mode = kModePlain;
    p.g.ab_fmt = 1;
    p.g.esize = 2;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.ps.init(static_cast<uint32_t>(M), static_cast<uint32_t>(N), tm, tn, sch.offset, sch.dir);
    p.g.num_kb = (K + 63) / 64;
    p.g.chunk_kb = kDequantChunkK / 64;
    p.g.total_tiles = static_cast<uint32_t>(tiles);
    p.g.C = static_cast<uint8_t*>(C);
    p.g.ldc = ldc;
    p.g.c_type = kOutBF16;
    p.g.c_vec = store_vec(C, ldc * 2, 0, 2);
    p.g.acc_vec = acc_out ? store_vec(acc_out, ldc * 4, 0, 4) : 4u;
    p.g.scale_a = scale_a;
    p.g.scale_b = scale_b;
    p.g.acc_out = acc_out;
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    const uint32_t ctas = sch.num_ctas ? sch.num_ctas : dev.sms;
    if (pair)
        return cuda_status(launch_pair_dequant(p, pair_grid(sch, tiles, dev.sms),
                                               stream));
    const uint32_t grid = static_cast<uint32_t>(std::min<uint64_t>(ctas, tiles));
    return cuda_status(launch_dequant(p, grid, stream));
}

size_t bst_gemm_grouped_quant_per_token_workspace_size(int32_t G, int64_t total_m, int64_t N, int64_t K) {
    if (G < 1 || total_m < 0 || N < 0 || K < 0) return 0;
    const size_t kp = static_cast<size_t>((K + 7) / 8 * 8);
    const size_t np = static_cast<size_t>((N + 7) / 8 * 8);
    const size_t a = static_cast<size_t>(total_m) * kp * 2;
    const size_t per_group = std::max(static_cast<size_t>(N) * kp, static_cast<size_t>(K) * np);
    return round256(a) + round256(static_cast<size_t>(G) * per_group * 2);
}

bst_status bst_gemm_grouped_quant_per_token(int32_t G, const int32_t* group_m, int64_t total_m, int64_t N, int64_t K,
                                            const int8_t* A, int64_t lda, const int8_t* B, bst_layout b_layout,
                                            int64_t ldb, int64_t stride_b, const float* scale_a, const float* scale_b,
                                            int64_t stride_sb, void* C, int64_t ldc, int32_t* acc_out,
                                            void* workspace, size_t workspace_bytes, const bst_sched* sched_in,
                                            void* stream_v) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || total_m < 0 || N < 0 || K < 0) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(total_m) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(K) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (b_layout != BST_ROW_MAJOR && b_layout != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    // 256 x 256 CTA-pair tiles only
    if ((sch.tile_m != 0 && sch.tile_m != 256) || (sch.tile_n != 0 && sch.tile_n != 256)) return BST_ERR_UNSUPPORTED;
    const bool b_kmajor = b_layout == BST_COL_MAJOR;   // each B_g stored [N, K]
    const int64_t b_rows = b_kmajor ? N : K, b_cols = b_kmajor ? K : N;
    if (ldc < N || ldc < 1 || lda < 1 || lda < K || ldb < 1 || ldb < b_cols) return BST_ERR_INVALID_ARG;
    if (G > 1 && (stride_b < b_rows * ldb || stride_sb < N)) return BST_ERR_INVALID_ARG;
    if (total_m == 0 || N == 0) return BST_OK;
    if (!group_m || !C || !scale_a || !scale_b || (K > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (K == 0) {
        cudaError_t e = launch_zero_fill(static_cast<uint8_t*>(C), ldc, 0, total_m, N, 1, 2, dev.sms, stream);
        if (e == cudaSuccess && acc_out)
            e = launch_zero_fill(reinterpret_cast<uint8_t*>(acc_out), ldc, 0, total_m, N, 1, 4, dev.sms, stream);
        return cuda_status(e);
    }
    const size_t need = bst_gemm_grouped_quant_per_token_workspace_size(G, total_m, N, K);
    if (!workspace || workspace_bytes < need) return BST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return BST_ERR_ALIGNMENT;
    const int64_t kp = (K + 7) / 8 * 8;
    const int64_t np = (N + 7) / 8 * 8;
    const int64_t per_group = std::max(N * kp, K * np);          // widened elements between groups
    uint16_t* wa = static_cast<uint16_t*>(workspace);
    uint16_t* wb = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) +
                                               round256(static_cast<size_t>(total_m) * kp * 2));
    const int64_t ldwb = b_kmajor ? kp : np;
    const uint64_t tiles_bound = ((total_m + 255) / 256 + G) * ((N + 255) / 256);
    if (tiles_bound >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    if (smem_pair_dequant() + 8 * (static_cast<uint32_t>(G) + 1) > dev.max_smem) return BST_ERR_UNSUPPORTED;

    const WidenArgs wa_args{A, lda, wa, kp, total_m, K};
    const WidenArgs wb_args{B, ldb, wb, ldwb, b_rows, b_cols, G, G > 1 ? stride_b : 0, per_group};
    if (launch_widen2_s8_bf16(wa_args, wb_args, dev.sms, stream, dev.err, timeout_ns()) != cudaSuccess)
        return BST_ERR_CUDA;

    OperandSpec a{wa, 2, static_cast<uint64_t>(total_m), static_cast<uint64_t>(K), kp, 0, 1, false};
    OperandSpec b{wb, 2, static_cast<uint64_t>(N), static_cast<uint64_t>(K), ldwb, per_group,
                  static_cast<uint64_t>(G), !b_kmajor};
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (bst_status s = fill_operand(p.g.a, &p.tmap_a, a, kBM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, true)) return s;
    if (bst_status s = fill_operand(p.g.b, &p.tmap_b, b, 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, true)) return s;
    p.g.M = 0; p.g.N = N; p.g.K = K;
    p.g.batch = 1;
    p.g.mode = kModeGrouped;
    p.g.ab_fmt = 1;
    p.g.esize = 2;
    p.g.swz_offset = sch.offset;
    p.g.swz_dir = sch.dir;
    p.g.num_kb = (K + 63) / 64;
    p.g.chunk_kb = kDequantChunkK / 64;
    p.g.group_m = group_m;
    p.g.G = static_cast<uint32_t>(G);
    p.g.total_m = static_cast<uint32_t>(total_m);
    p.g.C = static_cast<uint8_t*>(C);
    p.g.ldc = ldc;
    p.g.c_type = kOutBF16;
    p.g.c_vec = store_vec(C, ldc * 2, 0, 2);
    p.g.acc_vec = acc_out ? store_vec(acc_out, ldc * 4, 0, 4) : 4u;
    p.g.scale_a = scale_a;
    p.g.scale_b = scale_b;
    p.g.sb_group_stride = G > 1 ? stride_sb : 0;
    p.g.acc_out = acc_out;
    p.g.trace = sch.trace;
    p.g.timeline = sch.timeline;
    p.g.trace_cap = static_cast<uint32_t>(tiles_bound);
    p.g.err = dev.err;
    p.g.timeout_ns = timeout_ns();
    p.g.dynamic = sch.dynamic;
    p.g.shuffle_k = sch.shuffle_k;
    return cuda_status(launch_pair_dequant(p, pair_grid(sch, tiles_bound, dev.sms), stream));
}

size_t bst_gemm_grouped_slice_k_workspace_size(int32_t G) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups) return 0;
    return static_cast<size_t>(G) * 256 + round256(4 * (static_cast<size_t>(G) + 1));
}


bst_status bst_gemm_grouped_slice_k(int32_t G, const int32_t* group_k, int64_t M, int64_t N, int64_t total_k,
                                    const void* A, bst_layout a_layout, int64_t lda, const void* B,
                                    bst_layout b_layout, int64_t ldb, void* C, int64_t ldc, int64_t stride_c,
                                    bst_dtype ab_type, bst_dtype c_type, void* workspace, size_t workspace_bytes,
                                    const bst_sched* sched_in, void* stream_v) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || M < 0 || N < 0 || total_k < 0) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(M) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(total_k) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (ab_type != BST_F16 && ab_type != BST_BF16) return BST_ERR_UNSUPPORTED;
    uint32_t c_code;
    if (!out_code(c_type, c_code)) return BST_ERR_UNSUPPORTED;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if ((sch.tile_m != 0 && sch.tile_m != 256) || sch.split_k > 1) return BST_ERR_UNSUPPORTED;
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (G > 1 && stride_c < M * ldc) return BST_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BST_OK;
    if (!C || !group_k || (total_k > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    OperandSpec a, b;
    if (bst_status s = make_specs(M, N, total_k, A, a_layout, lda, 0, B, b_layout, ldb, 0, 2, 1, a, b)) return s;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const uint32_t csize = dtype_bytes(c_type);
    if (total_k == 0)   // every group is empty
        return cuda_status(launch_zero_fill(static_cast<uint8_t*>(C), ldc, stride_c, M, N, G, csize, dev.sms, stream));
    if (!tma_ok(a) || !tma_ok(b)) return BST_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < bst_gemm_grouped_slice_k_workspace_size(G)) return BST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return BST_ERR_ALIGNMENT;
    SliceKRun r;
    r.a = a;
    r.b = b;
    r.ab_fmt = ab_type == BST_BF16 ? 1u : 0u;
    r.dt = tmap_type(ab_type);
    r.c_code = c_code;
    r.csize = csize;
    r.C = C;
    r.ldc = ldc;
    r.stride_c = G > 1 ? stride_c : 0;
    return run_slice_k(r, G, group_k, M, N, total_k, static_cast<uint8_t*>(workspace), sch, dev, stream);
}

size_t bst_gemm_grouped_slice_k_quant_per_token_workspace_size(int32_t G, int64_t M, int64_t N, int64_t total_k) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || M < 0 || N < 0 || total_k < 0) return 0;
    const size_t kp = static_cast<size_t>((total_k + 7) / 8 * 8);
    const size_t mp = static_cast<size_t>((M + 7) / 8 * 8);
    const size_t np = static_cast<size_t>((N + 7) / 8 * 8);
    const size_t a = std::max(static_cast<size_t>(M) * kp, static_cast<size_t>(total_k) * mp) * 2;
    const size_t b = std::max(static_cast<size_t>(N) * kp, static_cast<size_t>(total_k) * np) * 2;
    return round256(bst_gemm_grouped_slice_k_workspace_size(G)) + round256(a) + round256(b);
}

bst_status bst_gemm_grouped_slice_k_quant_per_token(int32_t G, const int32_t* group_k, int64_t M, int64_t N,
                                                    int64_t total_k, const int8_t* A, bst_layout a_layout,
                                                    int64_t lda, const int8_t* B, bst_layout b_layout, int64_t ldb,
                                                    const float* scale_a, int64_t stride_sa, const float* scale_b,
                                                    int64_t stride_sb, void* C, int64_t ldc, int64_t stride_c,
                                                    int32_t* acc_out, void* workspace, size_t workspace_bytes,
                                                    const bst_sched* sched_in, void* stream_v) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || M < 0 || N < 0 || total_k < 0) return BST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(M) > kMaxDim || static_cast<uint64_t>(N) > kMaxDim ||
        static_cast<uint64_t>(total_k) > kMaxDim)
        return BST_ERR_INVALID_ARG;
    if (a_layout != BST_ROW_MAJOR && a_layout != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    if (b_layout != BST_ROW_MAJOR && b_layout != BST_COL_MAJOR) return BST_ERR_INVALID_ARG;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if ((sch.tile_m != 0 && sch.tile_m != 256) || (sch.tile_n != 0 && sch.tile_n != 256) || sch.split_k > 1)
        return BST_ERR_UNSUPPORTED;
    const bool a_kmajor = a_layout == BST_ROW_MAJOR;   // A stored [M, total_k]
    const bool b_kmajor = b_layout == BST_COL_MAJOR;   // B stored [N, total_k]
    if (ldc < N || ldc < 1) return BST_ERR_INVALID_ARG;
    if (lda < 1 || lda < (a_kmajor ? total_k : M) || ldb < 1 || ldb < (b_kmajor ? total_k : N))
        return BST_ERR_INVALID_ARG;
    if (G > 1 && (stride_c < M * ldc || stride_sa < 0 || stride_sb < 0)) return BST_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BST_OK;
    if (!C || !group_k || !scale_a || !scale_b || (total_k > 0 && (!A || !B))) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const int64_t sc = G > 1 ? stride_c : 0;
    if (total_k == 0) {
        cudaError_t e = launch_zero_fill(static_cast<uint8_t*>(C), ldc, sc, M, N, G, 2, dev.sms, stream);
        if (e == cudaSuccess && acc_out)
            e = launch_zero_fill(reinterpret_cast<uint8_t*>(acc_out), ldc, sc, M, N, G, 4, dev.sms, stream);
        return cuda_status(e);
    }
    if (!workspace || workspace_bytes < bst_gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, total_k))
        return BST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return BST_ERR_ALIGNMENT;
    const int64_t kp = (total_k + 7) / 8 * 8, mp = (M + 7) / 8 * 8, np = (N + 7) / 8 * 8;
    uint8_t* meta = static_cast<uint8_t*>(workspace);
    const size_t meta_bytes = round256(bst_gemm_grouped_slice_k_workspace_size(G));
    const size_t a_bytes = round256(std::max(static_cast<size_t>(M) * kp, static_cast<size_t>(total_k) * mp) * 2);
    uint16_t* wa = reinterpret_cast<uint16_t*>(meta + meta_bytes);
    uint16_t* wb = reinterpret_cast<uint16_t*>(meta + meta_bytes + a_bytes);
    const int64_t ldwa = a_kmajor ? kp : mp, ldwb = b_kmajor ? kp : np;
    const WidenArgs wa_args = a_kmajor ? WidenArgs{A, lda, wa, ldwa, M, total_k} : WidenArgs{A, lda, wa, ldwa, total_k, M};
    const WidenArgs wb_args = b_kmajor ? WidenArgs{B, ldb, wb, ldwb, N, total_k} : WidenArgs{B, ldb, wb, ldwb, total_k, N};
    if (launch_widen2_s8_bf16(wa_args, wb_args, dev.sms, stream, dev.err, timeout_ns()) != cudaSuccess)
        return BST_ERR_CUDA;
    SliceKRun r;
    r.a = OperandSpec{wa, 2, static_cast<uint64_t>(M), static_cast<uint64_t>(total_k), ldwa, 0, 1, !a_kmajor};
    r.b = OperandSpec{wb, 2, static_cast<uint64_t>(N), static_cast<uint64_t>(total_k), ldwb, 0, 1, !b_kmajor};
    r.ab_fmt = 1;
    r.dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    r.c_code = kOutBF16;
    r.csize = 2;
    r.C = C;
    r.ldc = ldc;
    r.stride_c = sc;
    r.scale_a = scale_a;
    r.scale_b = scale_b;
    r.stride_sa = G > 1 ? stride_sa : 0;
    r.stride_sb = G > 1 ? stride_sb : 0;
    r.acc_out = acc_out;
    r.dequant = true;
    return run_slice_k(r, G, group_k, M, N, total_k, meta, sch, dev, stream);
}

bst_status bst_swizzle_map(uint32_t M, uint32_t N, uint32_t tile_m, uint32_t tile_n, uint32_t batch,
                           const bst_sched* sched_in, uint32_t* out, void* stream) {
    if (tile_m < 1 || tile_n < 1 || batch < 1) return BST_ERR_INVALID_ARG;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if (M == 0 || N == 0) return BST_OK;
    if (!out) return BST_ERR_INVALID_ARG;
    const uint64_t lm = (static_cast<uint64_t>(M) + tile_m - 1) / tile_m;
    const uint64_t ln = (static_cast<uint64_t>(N) + tile_n - 1) / tile_n;
    const uint64_t total = lm * ln * batch;
    if (total >= (1ull << 32)) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    PlainSched s;
    s.init(M, N, tile_m, tile_n, sch.offset, sch.dir);
    return cuda_status(launch_swizzle_map(s, static_cast<uint32_t>(total), out, static_cast<cudaStream_t>(stream)));
}

bst_status bst_swizzle_map_grouped(int32_t G, const int32_t* group_m, uint32_t N, uint32_t tile_m, uint32_t tile_n,
                                   const bst_sched* sched_in, uint32_t* out, uint32_t max_tasks, void* stream) {
    if (G < 1 || static_cast<uint32_t>(G) > kMaxGroups || tile_m < 1 || tile_n < 1) return BST_ERR_INVALID_ARG;
    Sched sch;
    if (bst_status s = read_sched(sched_in, sch)) return s;
    if (N == 0) return BST_OK;
    if (!group_m || (!out && max_tasks > 0)) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    return cuda_status(launch_swizzle_map_grouped(group_m, static_cast<uint32_t>(G), N, tile_m, tile_n, sch.offset,
                                                  sch.dir, out, max_tasks, dev.err,
                                                  static_cast<cudaStream_t>(stream)));
}

bst_status bst_check_async(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BST_ERR_CUDA;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    uint32_t w[4] = {0, 0, 0, 0};
    if (cudaMemcpy(w, dev.err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BST_ERR_CUDA;
    if (w[0] == 0) return BST_OK;
    const uint32_t zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(dev.err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return BST_ERR_CUDA;
    return (w[0] & kErrTimeout) ? BST_ERR_TIMEOUT : BST_ERR_DEVICE;
}

const char* bst_status_string(bst_status s) {
    switch (s) {
        case BST_OK: return "ok";
        case BST_ERR_INVALID_ARG: return "invalid argument";
        case BST_ERR_UNSUPPORTED: return "unsupported dtype, layout or device";
        case BST_ERR_ALIGNMENT: return "address or stride not aligned for this path";
        case BST_ERR_CUDA: return "CUDA error";
        case BST_ERR_TIMEOUT: return "device-side wait timed out";
        case BST_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

void bst_set_wait_timeout_ns(uint64_t ns) { t_timeout_ns = ns; }

bst_status bst_wait_check(uint64_t timeout_ns, int32_t arrive, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return BST_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (bst_status s = device_info(dev)) return s;
    return cuda_status(launch_wait_check(timeout_ns, arrive ? 1u : 0u, dev.err, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
