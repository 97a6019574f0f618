// MXFP8 GEMM instantiations: e4m3 x e4m3 with one E8M0 scale per 32 K
// elements per row of A / column of B, tcgen05.mma kind::mxf8f6f4 with block
// scaling (the workload of "MI450 WMMA and ds_load Scheduling via a DAG
// Mutation", "An example run on a real kernel": float8_e4m3 A and B with MX
// scales).
#include "internal.h"

namespace bst {

template <uint32_t BN, uint32_t STAGES, uint32_t ACC>
static cudaError_t launch_one(const GemmParams& p, uint32_t grid, cudaStream_t stream) {
    using Lay = GemmLayout<BN, STAGES, ACC, kKindMXF8>;
    static_assert(Lay::smem_bytes(0) <= 232448, "shared memory per CTA");
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_kernel<BN, STAGES, ACC, kKindMXF8, kEpiStore>;
    const uint32_t smem = Lay::smem_bytes(0);
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, attr_done);
    if (e != cudaSuccess) return e;
    return launch_gemm(kern, p, grid, threads_for<kKindMXF8>(), smem, stream);
}

cudaError_t launch_mxf8(const GemmParams& p, uint32_t bn, uint32_t grid, cudaStream_t stream) {
    switch (bn) {
        case 128: return launch_one<128, kMxStages128, 2>(p, grid, stream);
        case 256: return launch_one<256, kMxStages256, 1>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

uint32_t smem_mxf8(uint32_t bn) {
    switch (bn) {
        case 128: return GemmLayout<128, kMxStages128, 2, kKindMXF8>::smem_bytes(0);
        case 256: return GemmLayout<256, kMxStages256, 1, kKindMXF8>::smem_bytes(0);
        default: return 0xFFFFFFFFu;
    }
}

}  // namespace bst
