// Debug map kernels that run the device scheduler of sched.cuh over every
// task index ("Block Scheduler Code Explained", section 7 execution flow:
// batch index, block coordinate, actual block shape per task), the
// zero-fill used when K == 0, and the self-check of the bounded waits.
#include "internal.h"

namespace bst {

// Plain / batched: the host-prepared scheduler the GEMM kernels use.
__global__ void swizzle_map_kernel(PlainSched s, uint32_t total, uint32_t* __restrict__ out) {
    for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t b, m, n, ma, na;
        s.coord(t, b, m, n, ma, na);
        uint32_t* o = out + static_cast<uint64_t>(t) * 5;
        o[0] = b;
        o[1] = m;
        o[2] = n;
        o[3] = ma;
        o[4] = na;
    }
}

cudaError_t launch_swizzle_map(const PlainSched& s, uint32_t total, uint32_t* out, cudaStream_t stream) {
    if (total == 0) return cudaSuccess;
    const uint32_t blocks = min((total + 255) / 256, 4096u);
    swizzle_map_kernel<<<blocks, 256, 0, stream>>>(s, total, out);
    return cudaGetLastError();
}

// One CTA: prefix sums of the group sizes in shared memory, then every
// thread walks task indices; the same GroupTable lookup and per-group
// re-targeted scheduler as the grouped GEMM.
__global__ void swizzle_map_grouped_kernel(const int32_t* __restrict__ group_m, uint32_t G, uint32_t N, uint32_t tm,
                                           uint32_t tn, uint32_t offset, uint32_t dir, uint32_t* __restrict__ out,
                                           uint32_t max_tasks, uint32_t* err) {
    __shared__ uint32_t tile_off[kMaxGroups + 1];
    __shared__ uint32_t row_off[kMaxGroups + 1];
    __shared__ uint32_t bad;
    if (threadIdx.x == 0) {
        const uint32_t loops_n = (N + tn - 1) / tn;
        tile_off[0] = 0;
        row_off[0] = 0;
        bad = 0;
        for (uint32_t g = 0; g < G; ++g) {
            int32_t mg = group_m[g];
            if (mg < 0) { bad = 1; mg = 0; }
            row_off[g + 1] = row_off[g] + static_cast<uint32_t>(mg);
            tile_off[g + 1] = tile_off[g] + ((static_cast<uint32_t>(mg) + tm - 1) / tm) * loops_n;
        }
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) atomicOr(&err[0], kErrGroups);
        return;
    }
    const uint32_t total = tile_off[G];
    if (total > max_tasks && threadIdx.x == 0) atomicOr(&err[0], kErrTraceOverflow);
    GroupTable gt{tile_off, row_off, G};
    for (uint32_t t = threadIdx.x; t < total && t < max_tasks; t += blockDim.x) {
        const uint32_t g = gt.find(t);
        SwizzleSched s;
        s.update(row_off[g + 1] - row_off[g], N, tm, tn, offset, dir);
        uint32_t m, n, ma, na;
        s.block_coord(t - tile_off[g], m, n);
        s.actual_shape(m, n, ma, na);
        uint32_t* o = out + static_cast<uint64_t>(t) * 5;
        o[0] = g;
        o[1] = m;
        o[2] = n;
        o[3] = ma;
        o[4] = na;
    }
}

cudaError_t launch_swizzle_map_grouped(const int32_t* group_m, uint32_t G, uint32_t N, uint32_t tile_m,
                                       uint32_t tile_n, uint32_t offset, uint32_t dir, uint32_t* out,
                                       uint32_t max_tasks, uint32_t* err, cudaStream_t stream) {
    swizzle_map_grouped_kernel<<<1, 256, 0, stream>>>(group_m, G, N, tile_m, tile_n, offset, dir, out, max_tasks,
                                                      err);
    return cudaGetLastError();
}

__global__ void zero_fill_kernel(uint8_t* C, int64_t ldc, int64_t batch_stride, int64_t rows, int64_t cols,
                                 int64_t batch, uint32_t esize) {
    const int64_t per = rows * cols;
    const int64_t total = per * batch;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / per;
        const int64_t rem = i - b * per;
        const int64_t r = rem / cols;
        const int64_t c = rem - r * cols;
        uint8_t* d = C + (b * batch_stride + r * ldc + c) * esize;
        for (uint32_t j = 0; j < esize; ++j) d[j] = 0;
    }
}

cudaError_t launch_zero_fill(uint8_t* C, int64_t ldc, int64_t batch_stride, int64_t rows, int64_t cols,
                             int64_t batch, uint32_t esize, uint32_t sms, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
    zero_fill_kernel<<<sms * 4, 256, 0, stream>>>(C, ldc, batch_stride, rows, cols, batch, esize);
    return cudaGetLastError();
}

// Self-check of the device-side failure detection: thread 0 waits on a
// shared-memory barrier with the same bounded wait the GEMM kernels use.  With
// arrive != 0 thread 32 arrives on it (the wait succeeds); otherwise nothing
// arrives, the wait gives up after timeout_ns and records a timeout in the
// error word.  Nothing asynchronous is in flight, so giving up is harmless.
__global__ void wait_check_kernel(uint64_t timeout_ns, uint32_t arrive, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 32 && arrive) mbar_arrive(&bar);
    if (threadIdx.x == 0) {
        const WaitCtl ctl{&abort_flag, timeout_ns, err};
        mbar_wait(&bar, 0, ctl, 99);
    }
}

cudaError_t launch_wait_check(uint64_t timeout_ns, uint32_t arrive, uint32_t* err, cudaStream_t stream) {
    wait_check_kernel<<<1, 64, 0, stream>>>(timeout_ns, arrive, err);
    return cudaGetLastError();
}

}  // namespace bst
