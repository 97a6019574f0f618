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

// BST_WIDEN_BULK=0 keeps the dense widening on ordinary loads and stores
static bool widen_bulk_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("BST_WIDEN_BULK");
        return !(e && e[0] == '0');
    }();
    return on;
}

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

// The dense widening as a bulk-copy stream: each CTA takes chunks of 16 KB of
// int8 (grid stride), one thread loads them with cp.async.bulk into a ring
// of four slots, the whole CTA converts a chunk into 32 KB of bf16 in shared
// memory, and the same thread stores it with a bulk copy.  Loads run four
// chunks ahead; a slot's output is refilled once its previous store has read
// it.  The last CTA widens the tail (fewer than 16 KB) with plain loads.  A
// wait for a chunk gives up after timeout_ns and records kErrTimeout.
constexpr uint32_t kWidenChunk = 16384;                 // int8 bytes per chunk
constexpr uint32_t kWidenSlots = 4;
constexpr uint32_t kWidenThreads = 256;
constexpr uint32_t kWidenSmem = kWidenSlots * (kWidenChunk + 2 * kWidenChunk) + kWidenSlots * 8;

struct WidenSeg {
    const int8_t* src;
    uint16_t* dst;
    uint64_t n;                                         // elements, a multiple of 16
};

// Both operands of a GEMM in one launch: the chunks of segment 0, then those
// of segment 1 (n = 0 for a single operand).
__global__ void __launch_bounds__(kWidenThreads, 1)
widen_s8_bf16_bulk_kernel(WidenSeg s0, WidenSeg s1, uint32_t* err, uint64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t* const in = sm;
    uint8_t* const out = sm + kWidenSlots * kWidenChunk;
    uint64_t* const full = reinterpret_cast<uint64_t*>(out + kWidenSlots * 2 * kWidenChunk);
    const uint64_t c0 = s0.n / kWidenChunk;
    const uint64_t nchunks = c0 + s1.n / kWidenChunk;
    // chunk c of the joint sequence: its source and destination
    auto chunk_src = [&](uint64_t c) { return c < c0 ? s0.src + c * kWidenChunk : s1.src + (c - c0) * kWidenChunk; };
    auto chunk_dst = [&](uint64_t c) { return c < c0 ? s0.dst + c * kWidenChunk : s1.dst + (c - c0) * kWidenChunk; };
    const uint64_t first = blockIdx.x, step = gridDim.x;
    const uint64_t mine = first < nchunks ? (nchunks - first + step - 1) / step : 0;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < kWidenSlots; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    auto load = [&](uint64_t i) {                       // thread 0: chunk i of this CTA into slot i % 4
        const uint32_t s = static_cast<uint32_t>(i % kWidenSlots);
        mbar_arrive_expect_tx(&full[s], kWidenChunk);
        bulk_load_global(in + s * kWidenChunk, chunk_src(first + i * step), kWidenChunk, &full[s]);
    };
    if (threadIdx.x == 0)
        for (uint64_t i = 0; i < kWidenSlots && i < mine; ++i) load(i);
    uint64_t i = 0;
    for (; i < mine; ++i) {
        const uint32_t s = static_cast<uint32_t>(i % kWidenSlots);
        const bool got = mbar_wait_drain(&full[s], static_cast<uint32_t>((i / kWidenSlots) & 1u), timeout_ns);
        if (__syncthreads_or(!got)) {
            if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
            break;
        }
        // the store that last read this output slot (chunk i - 4) has finished
        // reading it: at most three newer stores are still pending
        if (threadIdx.x == 0 && i >= kWidenSlots) bulk_wait_read_3();
        __syncthreads();
        const int4* q = reinterpret_cast<const int4*>(in + s * kWidenChunk);
        uint4* o = reinterpret_cast<uint4*>(out + s * 2 * kWidenChunk);
#pragma unroll
        for (uint32_t u = 0; u < kWidenChunk / 16 / kWidenThreads; ++u) {
            const uint32_t g = u * kWidenThreads + threadIdx.x;
            const int4 r = q[g];
            o[2 * g] = widen16_lo(r);
            o[2 * g + 1] = widen16_hi(r);
        }
        fence_proxy_async_smem();                       // generic writes -> the bulk store's reads
        __syncthreads();
        if (threadIdx.x == 0) {
            bulk_store_global(chunk_dst(first + i * step), out + s * 2 * kWidenChunk, 2 * kWidenChunk);
            bulk_commit_group();
            if (i + kWidenSlots < mine) load(i + kWidenSlots);
        }
    }
    if (threadIdx.x == 0) {
        bulk_wait_all();                                // the stores have completed
        // chunks loaded but not consumed (an abort) land before the CTA exits
        for (uint64_t j = i; j < mine && j < i + kWidenSlots; ++j)
            mbar_wait_drain(&full[j % kWidenSlots], static_cast<uint32_t>((j / kWidenSlots) & 1u), timeout_ns);
    }
    if (blockIdx.x == gridDim.x - 1) {
        // the tails: past each segment's last whole chunk, a multiple of 16 elements
        for (uint32_t k = 0; k < 2; ++k) {
            const WidenSeg& sg = k ? s1 : s0;
            const uint64_t t0 = sg.n / kWidenChunk * kWidenChunk / 16, t1 = sg.n / 16;
            const int4* s4 = reinterpret_cast<const int4*>(sg.src);
            uint4* d4 = reinterpret_cast<uint4*>(sg.dst);
            for (uint64_t g = t0 + threadIdx.x; g < t1; g += kWidenThreads) {
                const int4 r = __ldg(s4 + g);
                d4[2 * g] = widen16_lo(r);
                d4[2 * g + 1] = widen16_hi(r);
            }
        }
    }
}

static cudaError_t launch_widen_bulk(WidenSeg s0, WidenSeg s1, uint32_t sms, cudaStream_t stream, uint32_t* err,
                                     uint64_t timeout_ns) {
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(widen_s8_bf16_bulk_kernel), kWidenSmem, attr_done);
    if (e != cudaSuccess) return e;
    widen_s8_bf16_bulk_kernel<<<sms, kWidenThreads, kWidenSmem, stream>>>(s0, s1, err, timeout_ns);
    return cudaGetLastError();
}

// A dense operand (rows and batches back to back in source and destination,
// 16-byte aligned, whole 16-element groups): its element count, else 0.
static uint64_t dense_elems(const WidenArgs& w) {
    if (w.rows <= 0 || w.cols <= 0 || w.batch <= 0) return 0;
    const bool ok = reinterpret_cast<uintptr_t>(w.src) % 16 == 0 && reinterpret_cast<uintptr_t>(w.dst) % 16 == 0 &&
                    w.cols % 16 == 0 && w.ld_src == w.cols && w.ld_dst == w.cols &&
                    (w.batch == 1 || (w.bs_src == w.rows * w.cols && w.bs_dst == w.rows * w.cols));
    return ok ? static_cast<uint64_t>(w.rows) * w.cols * w.batch : 0u;
}

cudaError_t launch_widen2_s8_bf16(const WidenArgs& a, const WidenArgs& b, uint32_t sms, cudaStream_t stream,
                                  uint32_t* err, uint64_t timeout_ns) {
    const uint64_t na = dense_elems(a), nb = dense_elems(b);
    if (na && nb && err && na + nb >= 2ull * sms * kWidenChunk && widen_bulk_enabled())
        return launch_widen_bulk(WidenSeg{a.src, a.dst, na}, WidenSeg{b.src, b.dst, nb}, sms, stream, err, timeout_ns);
    cudaError_t e = launch_widen_s8_bf16(a.src, a.ld_src, a.dst, a.ld_dst, a.rows, a.cols, sms, stream, a.batch,
                                         a.bs_src, a.bs_dst, err, timeout_ns);
    if (e != cudaSuccess) return e;
    return launch_widen_s8_bf16(b.src, b.ld_src, b.dst, b.ld_dst, b.rows, b.cols, sms, stream, b.batch, b.bs_src,
                                b.bs_dst, err, timeout_ns);
}

cudaError_t launch_widen_s8_bf16(const int8_t* src, int64_t ld_src, uint16_t* dst, int64_t ld_dst, int64_t rows,
                                 int64_t cols, uint32_t sms, cudaStream_t stream, int64_t batch, int64_t bs_src,
                                 int64_t bs_dst, uint32_t* err, uint64_t timeout_ns) {
    if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
    const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (ld_src % 16 == 0) && (bs_src % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (ld_dst % 8 == 0) && (bs_dst % 8 == 0);
    const bool dense = vec && cols % 16 == 0 && ld_src == cols && ld_dst == cols &&
                       (batch == 1 || (bs_src == rows * cols && bs_dst == rows * cols));
    const uint64_t n = static_cast<uint64_t>(rows) * cols * batch;
    if (dense && err && n >= 2ull * sms * kWidenChunk && widen_bulk_enabled())
        return launch_widen_bulk(WidenSeg{src, dst, n}, WidenSeg{src, dst, 0}, sms, stream, err, timeout_ns);
    if (dense) {
        widen_s8_bf16_flat_kernel<<<sms * 4, 256, 0, stream>>>(src, dst, n / 16);
        return cudaGetLastError();
    }
    widen_s8_bf16_kernel<<<sms * 4, 256, 0, stream>>>(src, ld_src, bs_src, dst, ld_dst, bs_dst, rows, cols, batch, vec);
    return cudaGetLastError();
}

}  // namespace bst
