// MXFP8 GEMM instantiations: e4m3 x e4m3 with one E8M0 scale per 32 K
// elements per row of A / column of B, tcgen05.mma kind::mxf8f6f4 with block
// scaling (the workload of "MI450 WMMA and ds_load Scheduling via a DAG
// Mutation", "An example run on a real kernel": float8_e4m3 A and B with MX
// scales).
#include "gemm_pair_mx.cuh"
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

template <uint32_t BN, uint32_t STAGES, uint32_t S>
using MxSplit = OneCtaSplit<BN, STAGES, kKindMXF8, S>;

cudaError_t launch_mxf8_split(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream) {
    if (bn == 256 && splits == 2) return MxSplit<256, kMxSplitStages256, 2>::launch(p, tiles, stream);
    if (bn == 128 && splits == 2) return MxSplit<128, kMxStages128, 2>::launch(p, tiles, stream);
    if (bn == 128 && splits == 4) return MxSplit<128, kMxStages128, 4>::launch(p, tiles, stream);
    return cudaErrorInvalidValue;
}

// 0 when there is no such instantiation
cudaError_t mxf8_split_resident(uint32_t bn, uint32_t splits, uint32_t* out) {
    *out = 0;
    if (bn == 256 && splits == 2) return MxSplit<256, kMxSplitStages256, 2>::resident(out);
    if (bn == 128 && splits == 2) return MxSplit<128, kMxStages128, 2>::resident(out);
    if (bn == 128 && splits == 4) return MxSplit<128, kMxStages128, 4>::resident(out);
    return cudaSuccess;
}

// CTA pairs on 256 x BN tiles (no split of K): a persistent grid of as many
// clusters of 2 as fit at once, capped by the tiles.
template <uint32_t BN, uint32_t STAGES>
static cudaError_t launch_pair_mx_one(const GemmParams& p, uint32_t max_pairs, cudaStream_t stream) {
    using Lay = PairMxLayout<BN, STAGES>;
    static_assert(Lay::smem_bytes() <= 232448, "shared memory per CTA");
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_pair_mx_kernel<BN, STAGES>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), Lay::smem_bytes(), attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPairMxThreads);
    cfg.dynamicSmemBytes = Lay::smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> resident[64];
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int n = resident[dev & 63].load();
    if (n <= 0) {
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        resident[dev & 63].store(n);
    }
    cfg.gridDim = dim3(2 * std::max(1u, std::min(max_pairs, static_cast<uint32_t>(n))));
    add_pdl(cfg, attr);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_mxf8_pair(const GemmParams& p, uint32_t bn, uint32_t max_pairs, cudaStream_t stream) {
    switch (bn) {
        case 128: return launch_pair_mx_one<128, kPairMxStages128>(p, max_pairs, stream);
        case 256: return launch_pair_mx_one<256, kPairMxStages256>(p, max_pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

uint32_t smem_mxf8_pair(uint32_t bn) {
    switch (bn) {
        case 128: return PairMxLayout<128, kPairMxStages128>::smem_bytes();
        case 256: return PairMxLayout<256, kPairMxStages256>::smem_bytes();
        default: return 0xFFFFFFFFu;
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
