// Grouped slice-K set-up ("Block Dispatch Policies",
// 05_grouped_matmul_slice_k and 11_grouped_matmul_slice_k_per_token_dequant).
//
// Group g owns the K_g consecutive K indices [off_g, off_g + K_g) of A and B.
// Its K extent is ragged, so the GEMM cannot load it through the whole
// operand's tensor map: the last k-block of a group would read the next
// group's columns.  This kernel rewrites, per group, a copy of each
// operand's map on the device -- base moved to the group's first K element,
// K extent cut to K_g -- so TMA fills the group's tail with zeros exactly as
// it does at the edge of a matrix.  It also stores each group's k-block count
// and a status word (non-zero when the sizes are negative, overrun the
// operands' K, or leave a K-contiguous operand's group start off a 16-byte
// boundary), in which case the GEMM computes nothing and the error word is
// raised.
#include <cstring>

#include "internal.h"

namespace bst {

struct SliceKPrep {
    CUtensorMap tmpl_a;         // whole-operand maps (2-D)
    CUtensorMap tmpl_b;
    const int32_t* group_k;     // device [G]
    uint32_t G;
    uint64_t total_k;
    uint64_t a_base, b_base;    // global addresses of A and B
    uint64_t a_kstep, b_kstep;  // bytes from one K index to the next
    uint32_t a_kdim, b_kdim;    // map dimension that runs along K (0 or 1)
    uint8_t* maps;              // out: G x 256 bytes
    uint32_t* group_kb;         // out: G k-block counts, then the status
    uint32_t* err;
};

// Exclusive prefix sum of K_g over the warp's 32 groups starting at `base`,
// continuing from `carry`.  Negative sizes count as 0 and set *bad.
__device__ __forceinline__ uint64_t group_offset(const SliceKPrep& p, uint32_t g, uint64_t& carry, uint32_t& kg,
                                                 uint32_t& bad) {
    const uint32_t lane = threadIdx.x & 31u;
    int32_t v = g < p.G ? p.group_k[g] : 0;
    if (v < 0) { bad = 1; v = 0; }
    kg = static_cast<uint32_t>(v);
    uint64_t incl = kg;
#pragma unroll
    for (uint32_t d = 1; d < 32; d <<= 1) {
        const uint64_t r = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += r;
    }
    const uint64_t off = carry + incl - kg;
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    return off;
}

template <int KD>
__device__ __forceinline__ void write_group_map(uint8_t* slot, const CUtensorMap& tmpl, uint64_t addr, uint32_t kg) {
    const uint4* src = reinterpret_cast<const uint4*>(&tmpl);
    uint4* dst = reinterpret_cast<uint4*>(slot);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = src[i];
    tmap_replace_address(slot, addr);
    tmap_replace_dim<KD>(slot, kg);
}

// One warp.
__global__ void __launch_bounds__(32, 1) slice_k_prep_kernel(const __grid_constant__ SliceKPrep p) {
    const uint32_t lane = threadIdx.x & 31u;
    uint64_t carry = 0;
    uint32_t bad = 0;
    for (uint32_t base = 0; base < p.G; base += 32) {
        const uint32_t g = base + lane;
        uint32_t kg;
        const uint64_t off = group_offset(p, g, carry, kg, bad);
        if (g < p.G && kg > 0 && ((p.a_kdim == 0 && (off * p.a_kstep) % 16) || (p.b_kdim == 0 && (off * p.b_kstep) % 16)))
            bad = 1;
    }
    bad = __any_sync(0xFFFFFFFFu, bad) || carry > p.total_k;
    // maps only for consistent sizes (so none can reach past the operands)
    carry = 0;
    for (uint32_t base = 0; base < p.G; base += 32) {
        const uint32_t g = base + lane;
        uint32_t kg, dummy = 0;
        const uint64_t off = group_offset(p, g, carry, kg, dummy);
        if (g < p.G) {
            if (!bad && kg > 0) {
                uint8_t* slot = p.maps + static_cast<uint64_t>(g) * 256u;
                if (p.a_kdim == 0) write_group_map<0>(slot, p.tmpl_a, p.a_base + off * p.a_kstep, kg);
                else write_group_map<1>(slot, p.tmpl_a, p.a_base + off * p.a_kstep, kg);
                if (p.b_kdim == 0) write_group_map<0>(slot + 128, p.tmpl_b, p.b_base + off * p.b_kstep, kg);
                else write_group_map<1>(slot + 128, p.tmpl_b, p.b_base + off * p.b_kstep, kg);
            }
            p.group_kb[g] = bad ? 0u : (kg + 63u) / 64u;
        }
    }
    tmap_release();
    if (lane == 0) {
        p.group_kb[p.G] = bad;
        if (bad) atomicOr(&p.err[0], kErrGroups);
    }
}

cudaError_t launch_slice_k_prep(const CUtensorMap& tmpl_a, const CUtensorMap& tmpl_b, const int32_t* group_k,
                                uint32_t G, uint64_t total_k, const void* a, uint64_t a_kstep, uint32_t a_kdim,
                                const void* b, uint64_t b_kstep, uint32_t b_kdim, uint8_t* maps, uint32_t* group_kb,
                                uint32_t* err, cudaStream_t stream) {
    SliceKPrep p;
    std::memset(&p, 0, sizeof(p));
    p.tmpl_a = tmpl_a;
    p.tmpl_b = tmpl_b;
    p.group_k = group_k;
    p.G = G;
    p.total_k = total_k;
    p.a_base = reinterpret_cast<uint64_t>(a);
    p.b_base = reinterpret_cast<uint64_t>(b);
    p.a_kstep = a_kstep;
    p.b_kstep = b_kstep;
    p.a_kdim = a_kdim;
    p.b_kdim = b_kdim;
    p.maps = maps;
    p.group_kb = group_kb;
    p.err = err;
    slice_k_prep_kernel<<<1, 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace bst
