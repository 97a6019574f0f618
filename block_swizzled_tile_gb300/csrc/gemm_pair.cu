// CTA-pair (cta_group::2) fp16/bf16 GEMM instantiations and cluster launch.
#include "gemm_pair.cuh"
#include "internal.h"

namespace bst {

template <uint32_t BN, uint32_t STAGES, uint32_t EPI = kEpiStore>
static cudaError_t launch_pair_one(const GemmParams& p, uint32_t max_pairs, cudaStream_t stream) {
    using Lay = PairLayout<BN, STAGES, EPI>;
    static_assert(Lay::smem_bytes(kMaxGroups) <= 232448, "shared memory per CTA");
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_pair_kernel<BN, STAGES, EPI>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), Lay::smem_bytes(kMaxGroups), attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(pair_threads<EPI>());
    cfg.dynamicSmemBytes = Lay::smem_bytes((p.g.mode == kModeGrouped || p.g.mode == kModeSliceK) ? p.g.G : 0);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
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
    // dynamic tasks: one cluster per task (those that do not fit wait, and the
    // running ones cancel them to take their tasks); else a persistent grid
    if (p.g.dynamic && max_pairs > (1u << 30)) return cudaErrorInvalidValue;
    const uint32_t pairs = p.g.dynamic ? std::max(1u, max_pairs)
                                       : std::max(1u, std::min(max_pairs, static_cast<uint32_t>(n)));
    cfg.gridDim = dim3(2 * pairs);
    add_pdl(cfg, attr);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_pair(const GemmParams& p, uint32_t bn, uint32_t max_pairs, cudaStream_t stream) {
    switch (bn) {
        case 128: return launch_pair_one<128, kPairStages128>(p, max_pairs, stream);
        case 256: return launch_pair_one<256, kPairStages256>(p, max_pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Ring depth of each split-K instantiation: what is left of the shared
// memory after the receive slots and the epilogue staging.
template <uint32_t BN, uint32_t S>
struct SplitStages;
template <> struct SplitStages<256, 2> { static constexpr uint32_t value = 4; };
template <> struct SplitStages<128, 2> { static constexpr uint32_t value = 7; };
template <> struct SplitStages<256, 4> { static constexpr uint32_t value = 3; };
template <> struct SplitStages<128, 4> { static constexpr uint32_t value = 6; };

template <uint32_t BN, uint32_t S>
struct SplitLaunch {
    static constexpr uint32_t kStages = SplitStages<BN, S>::value;
    using Lay = SplitLayout<BN, kStages, S>;
    static constexpr auto kern = gemm_pair_splitk_kernel<BN, kStages, S>;

    static cudaLaunchConfig_t config(uint32_t tiles, cudaStream_t stream, cudaLaunchAttribute* attr) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * S * tiles);
        cfg.blockDim = dim3(Lay::kThreads);
        cfg.dynamicSmemBytes = Lay::smem_bytes();
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
        return set_smem_once(reinterpret_cast<const void*>(kern), Lay::smem_bytes(), attr_done);
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
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = config(tiles, stream, attr);
        add_pdl(cfg, attr);
        return cudaLaunchKernelEx(&cfg, kern, p);
    }
};

cudaError_t launch_pair_splitk(const GemmParams& p, uint32_t bn, uint32_t splits, uint32_t tiles, cudaStream_t stream) {
    if (bn == 256 && splits == 2) return SplitLaunch<256, 2>::launch(p, tiles, stream);
    if (bn == 128 && splits == 2) return SplitLaunch<128, 2>::launch(p, tiles, stream);
    if (bn == 256 && splits == 4) return SplitLaunch<256, 4>::launch(p, tiles, stream);
    if (bn == 128 && splits == 4) return SplitLaunch<128, 4>::launch(p, tiles, stream);
    return cudaErrorInvalidValue;
}

cudaError_t splitk_resident_clusters(uint32_t bn, uint32_t splits, uint32_t* out) {
    if (bn == 256 && splits == 2) return SplitLaunch<256, 2>::resident(out);
    if (bn == 128 && splits == 2) return SplitLaunch<128, 2>::resident(out);
    if (bn == 256 && splits == 4) return SplitLaunch<256, 4>::resident(out);
    if (bn == 128 && splits == 4) return SplitLaunch<128, 4>::resident(out);
    return cudaErrorInvalidValue;
}

uint32_t smem_splitk(uint32_t bn, uint32_t splits) {
    if (bn == 256 && splits == 2) return SplitLaunch<256, 2>::Lay::smem_bytes();
    if (bn == 128 && splits == 2) return SplitLaunch<128, 2>::Lay::smem_bytes();
    if (bn == 256 && splits == 4) return SplitLaunch<256, 4>::Lay::smem_bytes();
    if (bn == 128 && splits == 4) return SplitLaunch<128, 4>::Lay::smem_bytes();
    return 0;
}

cudaError_t launch_pair_dequant(const GemmParams& p, uint32_t max_pairs, cudaStream_t stream) {
    return launch_pair_one<256, kPairDequantStages, kEpiDequant>(p, max_pairs, stream);
}

uint32_t smem_pair_dequant() { return PairLayout<256, kPairDequantStages, kEpiDequant>::smem_bytes(0); }

uint32_t smem_pair(uint32_t bn, uint32_t groups) {
    switch (bn) {
        case 128: return PairLayout<128, kPairStages128>::smem_bytes(groups);
        case 256: return PairLayout<256, kPairStages256>::smem_bytes(groups);
        default: return 0xFFFFFFFFu;
    }
}

}  // namespace bst
