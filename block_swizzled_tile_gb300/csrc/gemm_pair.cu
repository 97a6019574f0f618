// CTA-pair (cta_group::2) fp16/bf16 GEMM instantiations and cluster launch.
#include "gemm_pair.cuh"
#include "internal.h"

namespace bst {

template <uint32_t BN, uint32_t STAGES>
static cudaError_t launch_pair_one(const GemmParams& p, uint32_t max_pairs, cudaStream_t stream) {
    using Lay = PairLayout<BN, STAGES>;
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_pair_kernel<BN, STAGES>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), Lay::smem_bytes(kMaxGroups), attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kNumThreads);
    cfg.dynamicSmemBytes = Lay::smem_bytes(p.g.mode == kModeGrouped ? p.g.G : 0);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many pairs as can be resident at once (once per device), capped by the work
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
    const uint32_t pairs = std::max(1u, std::min(max_pairs, static_cast<uint32_t>(n)));
    cfg.gridDim = dim3(2 * pairs);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_pair(const GemmParams& p, uint32_t bn, uint32_t max_pairs, cudaStream_t stream) {
    switch (bn) {
        case 128: return launch_pair_one<128, kPairStages128>(p, max_pairs, stream);
        case 256: return launch_pair_one<256, kPairStages256>(p, max_pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <uint32_t S>
struct SplitLaunch {
    using Lay = PairLayout<256, kPairStages256>;
    static constexpr auto kern = gemm_pair_splitk_kernel<256, kPairStages256, S>;

    static cudaLaunchConfig_t config(uint32_t tiles, cudaStream_t stream, cudaLaunchAttribute* attr) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * S * tiles);
        cfg.blockDim = dim3(kNumThreads);
        cfg.dynamicSmemBytes = Lay::smem_bytes(0);
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2 * S;
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

    // clusters of 2*S CTAs that can be resident at once on the current device
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
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = config(tiles, stream, attr);
        return cudaLaunchKernelEx(&cfg, kern, p);
    }
};

cudaError_t launch_pair_splitk(const GemmParams& p, uint32_t splits, uint32_t tiles, cudaStream_t stream) {
    switch (splits) {
        case 2: return SplitLaunch<2>::launch(p, tiles, stream);
        case 4: return SplitLaunch<4>::launch(p, tiles, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t splitk_resident_clusters(uint32_t splits, uint32_t* out) {
    switch (splits) {
        case 2: return SplitLaunch<2>::resident(out);
        case 4: return SplitLaunch<4>::resident(out);
        default: return cudaErrorInvalidValue;
    }
}

uint32_t smem_pair(uint32_t bn, uint32_t groups) {
    switch (bn) {
        case 128: return PairLayout<128, kPairStages128>::smem_bytes(groups);
        case 256: return PairLayout<256, kPairStages256>::smem_bytes(groups);
        default: return 0xFFFFFFFFu;
    }
}

}  // namespace bst
