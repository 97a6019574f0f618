// bst_gemm_quant_per_token_noalloc: the int8 per-token-dequant GEMM with its
// bf16 operand scratch taken from a fixed array compiled into this library,
// so that the call allocates no device memory of any kind.
//
// The array lives in device global memory of every device that loads the
// library (BST_NOALLOC_SCRATCH_BYTES each).  Its device address is looked up
// with cudaGetSymbolAddress the first time the entry point runs on a device,
// with that device current, and kept for the life of the process; after a
// cudaDeviceReset of that device the kept address is stale.  Nothing in the
// scratch has to start at zero: the call writes every scratch byte it reads
// (the widened operands) before its GEMM kernel reads it.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "bst.h"

// File-scope scratch array with internal linkage; host code never uses its
// name as an address, only the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BST_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];

// The scratch array's device address on the current device (set up once per
// device).  Returns 0 on a CUDA error.
uintptr_t scratch_address(bst_status* st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { *st = BST_ERR_CUDA; return 0; }
    if (dev < 0 || dev >= kMaxDevices) { *st = BST_ERR_UNSUPPORTED; return 0; }
    uintptr_t addr = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (addr) return addr;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) { *st = BST_ERR_CUDA; return 0; }
    addr = reinterpret_cast<uintptr_t>(p);
    g_scratch_addr[dev].store(addr, std::memory_order_release);
    return addr;
}

}  // namespace

extern "C" bst_status bst_gemm_quant_per_token_noalloc(int64_t M, int64_t N, int64_t K, const int8_t* A, int64_t lda,
                                                       const int8_t* B, bst_layout b_layout, int64_t ldb,
                                                       const float* scale_a, const float* scale_b, void* C,
                                                       int64_t ldc, int32_t* acc_out, const bst_sched* sched,
                                                       void* stream) {
    if (M < 0 || N < 0 || K < 0) return BST_ERR_INVALID_ARG;
    // rejected before any CUDA call: the problem's scratch would not fit
    if (bst_gemm_quant_per_token_workspace_size(M, N, K) > BST_NOALLOC_SCRATCH_BYTES) return BST_ERR_UNSUPPORTED;
    bst_status st = BST_OK;
    const uintptr_t scratch = scratch_address(&st);
    if (!scratch) return st;
    return bst_gemm_quant_per_token(M, N, K, A, lda, B, b_layout, ldb, scale_a, scale_b, C, ldc, acc_out,
                                    reinterpret_cast<void*>(scratch), BST_NOALLOC_SCRATCH_BYTES, sched, stream);
}
