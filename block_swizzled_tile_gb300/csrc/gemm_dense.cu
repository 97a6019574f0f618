// fp16 / bf16 GEMM instantiations (plain, batched and grouped share them; the
// mode is a run-time field of GemmParams).
#include "internal.h"

namespace bst {

template <uint32_t BN, uint32_t STAGES>
static cudaError_t launch_one(const GemmParams& p, uint32_t grid, cudaStream_t stream) {
    using Lay = GemmLayout<BN, STAGES, 2, kKindF16>;
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_kernel<BN, STAGES, 2, kKindF16, kEpiStore>;
    // BN 64 also serves B through the two-row view, whose staging takes the
    // place of the group table
    constexpr uint32_t kMax = (BN == 64 && Lay::smem_bytes_rows2() > Lay::smem_bytes(kMaxGroups))
                                  ? Lay::smem_bytes_rows2() : Lay::smem_bytes(kMaxGroups);
    static_assert(kMax <= 232448, "shared memory per CTA");
    if (p.g.b.rows2 && BN != 64) return cudaErrorInvalidValue;
    const uint32_t smem = p.g.b.rows2 ? Lay::smem_bytes_rows2() : Lay::smem_bytes(p.g.mode == kModeGrouped ? p.g.G : 0);
    // the limit is set once for the largest group table (or staging) any call can need
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), kMax, attr_done);
    if (e != cudaSuccess) return e;
    return launch_gemm(kern, p, grid, threads_for<kKindF16>(), smem, stream);
}

cudaError_t launch_dense(const GemmParams& p, uint32_t bn, uint32_t grid, cudaStream_t stream) {
    switch (bn) {
        case 64: return launch_one<64, kDenseStages64>(p, grid, stream);
        case 128: return launch_one<128, kDenseStages128>(p, grid, stream);
        case 256: return launch_one<256, kDenseStages256>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

uint32_t smem_dense_rows2() { return GemmLayout<64, kDenseStages64, 2, kKindF16>::smem_bytes_rows2(); }

uint32_t smem_dense(uint32_t bn, uint32_t groups) {
    switch (bn) {
        case 64: return GemmLayout<64, kDenseStages64, 2, kKindF16>::smem_bytes(groups);
        case 128: return GemmLayout<128, kDenseStages128, 2, kKindF16>::smem_bytes(groups);
        case 256: return GemmLayout<256, kDenseStages256, 2, kKindF16>::smem_bytes(groups);
        default: return 0xFFFFFFFFu;
    }
}

template <uint32_t BN, uint32_t S>
using DenseSplit = OneCtaSplit<BN, BN == 64 ? kDenseStages64 : kDenseStages128, kKindF16, S>;

cudaError_t launch_dense_split(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream) {
    if (bn == 64 && splits == 2) return DenseSplit<64, 2>::launch(p, tiles, stream);
    if (bn == 128 && splits == 2) return DenseSplit<128, 2>::launch(p, tiles, stream);
    if (bn == 128 && splits == 4) return DenseSplit<128, 4>::launch(p, tiles, stream);
    return cudaErrorInvalidValue;
}

// 0 when there is no such instantiation
cudaError_t dense_split_resident(uint32_t bn, uint32_t splits, uint32_t* out) {
    *out = 0;
    if (bn == 64 && splits == 2) return DenseSplit<64, 2>::resident(out);
    if (bn == 128 && splits == 2) return DenseSplit<128, 2>::resident(out);
    if (bn == 128 && splits == 4) return DenseSplit<128, 4>::resident(out);
    return cudaSuccess;
}

uint32_t smem_dense_split(uint32_t bn, uint32_t splits) {
    if (bn == 64 && splits == 2) return DenseSplit<64, 2>::Lay::smem_bytes(0);
    if (bn == 128 && splits == 2) return DenseSplit<128, 2>::Lay::smem_bytes(0);
    if (bn == 128 && splits == 4) return DenseSplit<128, 4>::Lay::smem_bytes(0);
    return 0xFFFFFFFFu;
}

}  // namespace bst
