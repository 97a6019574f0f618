// int8 GEMM with per-token dequant ("Block Dispatch Policies",
// 12_quant_matmul).
//
// sm_103a has no int8 tcgen05 MMA, so the product is formed exactly on the
// bf16 tensor cores: every int8 value is exact in bf16, every product of two
// (|p| <= 127*127 = 16129) is exact in fp32, and a sum of at most 1024 of them
// stays below 1024*16129 < 2^24, where every integer is exact in fp32.  The
// MMA therefore accumulates K-chunks of 1024 in TMEM; the epilogue converts
// each chunk to int32 and carries the running sum in registers, then applies
// scale_a[row] * scale_b[col] once at the end.
#include "internal.h"

namespace bst {

cudaError_t launch_dequant(const GemmParams& p, uint32_t grid, cudaStream_t stream) {
    using Lay = GemmLayout<128, kDequantStages, 2, kKindF16>;
    static std::atomic<uint64_t> attr_done{0};
    auto kern = gemm_kernel<128, kDequantStages, 2, kKindF16, kEpiDequant>;
    const uint32_t smem = Lay::smem_bytes(0);
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, attr_done);
    if (e != cudaSuccess) return e;
    return launch_gemm(kern, p, grid, threads_for<kKindF16>(), smem, stream);
}

uint32_t smem_dequant() { return GemmLayout<128, kDequantStages, 2, kKindF16>::smem_bytes(0); }

// Widens int8 to bf16, 16 elements per thread per step when the rows allow
// 16-byte loads, element by element otherwise.  Bandwidth bound.
__global__ void widen_s8_bf16_kernel(const int8_t* __restrict__ src, int64_t ld_src, int64_t bs_src,
                                     uint16_t* __restrict__ dst, int64_t ld_dst, int64_t bs_dst, int64_t rows,
                                     int64_t cols, int64_t batch, int vec) {
    // rows of all batches in one index space: global row R = b * rows + r
    const int64_t all_rows = rows * batch;
    const int64_t chunks_per_row = vec ? cols / 16 : 0;
    const int64_t total_vec = all_rows * chunks_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total_vec; i += stride) {
        const int64_t R = i / chunks_per_row;
        const int64_t c = (i - R * chunks_per_row) * 16;
        const int64_t b = R / rows, r = R - b * rows;
        const int4 raw = __ldg(reinterpret_cast<const int4*>(src + b * bs_src + r * ld_src + c));
        const int8_t* q = reinterpret_cast<const int8_t*>(&raw);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(q[2 * j]), static_cast<float>(q[2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint4* d = reinterpret_cast<uint4*>(dst + b * bs_dst + r * ld_dst + c);
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    // columns not covered by 16-wide chunks
    const int64_t tail0 = chunks_per_row * 16;
    const int64_t tail_cols = cols - tail0;
    const int64_t total_tail = all_rows * tail_cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total_tail; i += stride) {
        const int64_t R = i / tail_cols;
        const int64_t c = tail0 + (i - R * tail_cols);
        const int64_t b = R / rows, r = R - b * rows;
        const __nv_bfloat16 h = __float2bfloat16_rn(static_cast<float>(src[b * bs_src + r * ld_src + c]));
        dst[b * bs_dst + r * ld_dst + c] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

__device__ __forceinline__ uint4 widen16_lo(const int4& raw) {
    const int8_t* q = reinterpret_cast<const int8_t*>(&raw);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(q[2 * j]), static_cast<float>(q[2 * j + 1]));
        w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 widen16_hi(const int4& raw) {
    const int8_t* q = reinterpret_cast<const int8_t*>(&raw) + 8;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(q[2 * j]), static_cast<float>(q[2 * j + 1]));
        w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The same for a dense operand (rows, and batches, back to back in both the
// source and the destination): one flat array of n16 chunks of 16 elements,
// no index division, four 16-byte loads in flight per thread.
__global__ void widen_s8_bf16_flat_kernel(const int8_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t n16) {
    const int4* s = reinterpret_cast<const int4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        int4 r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) r[u] = __ldg(s + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            d[2 * (i + u * stride)] = widen16_lo(r[u]);
            d[2 * (i + u * stride) + 1] = widen16_hi(r[u]);
        }
    }
    for (; i < n16; i += stride) {
        const int4 r = __ldg(s + i);
        d[2 * i] = widen16_lo(r);
        d[2 * i + 1] = widen16_hi(r);
    }
}

cudaError_t launch_widen_s8_bf16(const int8_t* src, int64_t ld_src, uint16_t* dst, int64_t ld_dst, int64_t rows,
                                 int64_t cols, uint32_t sms, cudaStream_t stream, int64_t batch, int64_t bs_src,
                                 int64_t bs_dst) {
    if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
    const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (ld_src % 16 == 0) && (bs_src % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (ld_dst % 8 == 0) && (bs_dst % 8 == 0);
    const bool dense = vec && cols % 16 == 0 && ld_src == cols && ld_dst == cols &&
                       (batch == 1 || (bs_src == rows * cols && bs_dst == rows * cols));
    if (dense) {
        widen_s8_bf16_flat_kernel<<<sms * 4, 256, 0, stream>>>(src, dst, rows * cols * batch / 16);
        return cudaGetLastError();
    }
    widen_s8_bf16_kernel<<<sms * 4, 256, 0, stream>>>(src, ld_src, bs_src, dst, ld_dst, bs_dst, rows, cols, batch, vec);
    return cudaGetLastError();
}

}  // namespace bst
