// Host-side interface between the C-ABI layer (api.cu) and the translation
// units that instantiate the kernels.  Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "gemm_kernel.cuh"

namespace bst {

// Raises a kernel's dynamic shared-memory limit once per device (bit `dev`
// of `done`), so that later launches -- including ones recorded into a CUDA
// graph -- make no attribute call.
inline cudaError_t set_smem_once(const void* kern, uint32_t bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Programmatic dependent launch for the GEMM kernels (all of which execute
// griddepcontrol.wait before their first global-memory access): the next
// kernel's launch and shared-memory / TMEM set-up overlap the tail of the
// previous one.  On unless the environment sets BST_PDL=0.
inline bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("BST_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Appends the programmatic-serialization attribute to `cfg` (attrs must have
// room for one more entry).
inline void add_pdl(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attrs) {
    if (!pdl_enabled()) return;
    cudaLaunchAttribute& a = attrs[cfg.numAttrs];
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    ++cfg.numAttrs;
}

// Launches a one-CTA GEMM kernel: `grid` CTAs of `threads` threads.
template <typename Kern>
inline cudaError_t launch_gemm(Kern kern, const GemmParams& p, uint32_t grid, uint32_t threads, uint32_t smem,
                               cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    add_pdl(cfg, attrs);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Split-K of one-CTA tiles: clusters of S CTAs, one 128 x BN tile per
// cluster, K divided among the cluster's CTAs and the partials summed
// through distributed shared memory.
template <uint32_t BN, uint32_t STAGES, uint32_t KIND, uint32_t S>
struct OneCtaSplit {
    using Lay = GemmLayout<BN, STAGES, 1, KIND, S>;
    static_assert(Lay::smem_bytes(0) <= 232448, "shared memory per CTA");
    static constexpr auto kern = gemm_kernel<BN, STAGES, 1, KIND, kEpiStore, S>;

    static cudaLaunchConfig_t config(uint32_t tiles, cudaStream_t stream, cudaLaunchAttribute* attr) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(S * tiles);
        cfg.blockDim = dim3(threads_for<KIND>());
        cfg.dynamicSmemBytes = Lay::smem_bytes(0);
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cfg;
    }
    static cudaError_t prepare() {
        static std::atomic<uint64_t> attr_done{0};
        return set_smem_once(reinterpret_cast<const void*>(kern), Lay::smem_bytes(0), attr_done);
    }
    // clusters of S that can be resident at once
    static cudaError_t resident(uint32_t* out) {
        static std::atomic<int> cache[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        int n = cache[dev & 63].load();
        if (n <= 0) {
            if ((e = prepare()) != cudaSuccess) return e;
            cudaLaunchAttribute attr[1];
            cudaLaunchConfig_t cfg = config(1, nullptr, attr);
            if ((e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg)) != cudaSuccess)
                return e;
            cache[dev & 63].store(n);
        }
        *out = n > 0 ? static_cast<uint32_t>(n) : 0u;
        return cudaSuccess;
    }
    static cudaError_t launch(const GemmParams& p, uint32_t tiles, cudaStream_t stream) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = config(tiles, stream, attr);
        add_pdl(cfg, attr);
        return cudaLaunchKernelEx(&cfg, kern, p);
    }
};

// Kernel launches.  Each returns the cudaError_t of the launch (attribute
// setting included); `grid` CTAs of kNumThreads threads on `stream`.
cudaError_t launch_dense(const GemmParams& p, uint32_t bn, uint32_t grid, cudaStream_t stream);
// fp16 / bf16 one-CTA split-K (operands that TMA cannot fetch): bn 64 with 2
// splits, bn 128 with 2 or 4
cudaError_t launch_dense_split(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream);
cudaError_t dense_split_resident(uint32_t bn, uint32_t splits, uint32_t* out);
uint32_t smem_dense_split(uint32_t bn, uint32_t splits);
cudaError_t launch_mxf8(const GemmParams& p, uint32_t bn, uint32_t grid, cudaStream_t stream);
// MXFP8 split-K over clusters of `splits` CTAs (tile 128 x bn), one tile per cluster
cudaError_t launch_mxf8_split(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream);
// MXFP8 on CTA-pair tiles 256 x bn (no split): clusters of 2, at most max_pairs
cudaError_t launch_mxf8_pair(const GemmParams& p, uint32_t bn, uint32_t max_pairs, cudaStream_t stream);
uint32_t smem_mxf8_pair(uint32_t bn);
// clusters the MXFP8 split-K kernel keeps resident at once (0: no such shape)
cudaError_t mxf8_split_resident(uint32_t bn, uint32_t splits, uint32_t* out);
cudaError_t launch_dequant(const GemmParams& p, uint32_t grid, cudaStream_t stream);
// CTA-pair kernel: launches clusters of 2, at most max_pairs of them (and no
// more than fit on the device at once)
cudaError_t launch_pair(const GemmParams& p, uint32_t bn, uint32_t max_pairs, cudaStream_t stream);
// split-K CTA pairs on 256 x 256 tiles: one cluster of 2*splits CTAs per tile
cudaError_t launch_pair_splitk(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream);
// int8 per-token dequant on 256 x 256 CTA-pair tiles (bf16-widened operands)
cudaError_t launch_pair_dequant(const GemmParams& p, uint32_t max_pairs, cudaStream_t stream);
uint32_t smem_pair_dequant();
// clusters of 2*splits CTAs the split-K kernel (tile 256 x bn) can keep resident at once
cudaError_t splitk_resident_clusters(uint32_t bn, uint32_t splits, uint32_t* out);
// dynamic shared memory of the split-K kernel (0: no such instantiation)
uint32_t smem_splitk(uint32_t bn, uint32_t splits);

// Shared-memory bytes a launch needs (for validation of the device limit).
uint32_t smem_dense(uint32_t bn, uint32_t groups);
uint32_t smem_dense_rows2();   // BN 64 with B through the two-row view
uint32_t smem_mxf8(uint32_t bn);
uint32_t smem_dequant();
uint32_t smem_pair(uint32_t bn, uint32_t groups);

// int8 [rows, cols] (ld_src elements) -> bf16 [rows, cols] (ld_dst elements)
// One int8 operand to widen into a bf16 copy (leading dimensions and batch
// strides in elements).
struct WidenArgs {
    const int8_t* src;
    int64_t ld_src;
    uint16_t* dst;
    int64_t ld_dst;
    int64_t rows, cols;
    int64_t batch = 1, bs_src = 0, bs_dst = 0;
};

// Both operands of an int8 GEMM: one bulk-copy launch when both are dense,
// else one launch each.
cudaError_t launch_widen2_s8_bf16(const WidenArgs& a, const WidenArgs& b, uint32_t sms, cudaStream_t stream,
                                  uint32_t* err, uint64_t timeout_ns);

// err / timeout_ns: the device error word and the wait limit of the bulk-copy
// widening (large dense operands); without err the ordinary-load kernels run
cudaError_t launch_widen_s8_bf16(const int8_t* src, int64_t ld_src, uint16_t* dst, int64_t ld_dst, int64_t rows,
                                 int64_t cols, uint32_t sms, cudaStream_t stream, int64_t batch = 1,
                                 int64_t bs_src = 0, int64_t bs_dst = 0, uint32_t* err = nullptr,
                                 uint64_t timeout_ns = 0);

// grouped slice-K: per-group tensor maps (G x 256 bytes at `maps`) and
// k-block counts plus a status word (G + 1 words at `group_kb`), from the
// whole-operand maps; a_kstep / b_kstep are the bytes between consecutive K
// indices and a_kdim / b_kdim the map dimension along K
cudaError_t launch_slice_k_prep(const CUtensorMap& tmpl_a, const CUtensorMap& tmpl_b, const int32_t* group_k,
                                uint32_t G, uint64_t total_k, const void* a, uint64_t a_kstep, uint32_t a_kdim,
                                const void* b, uint64_t b_kstep, uint32_t b_kdim, uint8_t* maps, uint32_t* group_kb,
                                uint32_t* err, cudaStream_t stream);

// zero an [rows, cols] row-major output of `esize`-byte elements, `batch`
// times at `batch_stride` elements apart
cudaError_t launch_zero_fill(uint8_t* C, int64_t ldc, int64_t batch_stride, int64_t rows, int64_t cols,
                             int64_t batch, uint32_t esize, uint32_t sms, cudaStream_t stream);

cudaError_t launch_swizzle_map(const PlainSched& s, uint32_t total, uint32_t* out, cudaStream_t stream);
cudaError_t launch_wait_check(uint64_t timeout_ns, uint32_t arrive, uint32_t* err, cudaStream_t stream);
cudaError_t launch_swizzle_map_grouped(const int32_t* group_m, uint32_t G, uint32_t N, uint32_t tile_m,
                                       uint32_t tile_n, uint32_t offset, uint32_t dir, uint32_t* out,
                                       uint32_t max_tasks, uint32_t* err, cudaStream_t stream);

// Configurations instantiated for each kernel family.
constexpr uint32_t kDenseStages64 = 7, kDenseStages128 = 6, kDenseStages256 = 4;
constexpr uint32_t kMxStages128 = 6, kMxStages256 = 3;
// split-K tiles stage their epilogue stores in the idle ring, so 128 x 256
// split tiles fit a fourth stage (more bytes in flight per SM)
constexpr uint32_t kMxSplitStages256 = 4;
constexpr uint32_t kDequantStages = 6;
constexpr uint32_t kPairStages128 = 8, kPairStages256 = 6;
constexpr uint32_t kPairDequantStages = 5;
constexpr uint32_t kPairMxStages128 = 7, kPairMxStages256 = 4;
constexpr uint32_t kDequantChunkK = 1024;  // K elements per exact fp32 chunk

}  // namespace bst
