"""Python binding of the bst C ABI (include/bst.h): argument marshalling only.

Every function here has the name and argument order of its C counterpart
(minus the ``bst_`` prefix).  Pointer arguments accept a torch tensor (its
``data_ptr()``), an int address or None; ``stream`` defaults to torch's
current CUDA stream.  A non-OK status raises ``BstError``.  All arithmetic
runs in the CUDA kernels of ``libbst.so``; if the library is missing the
import of any entry point fails loudly -- there is no fallback.
"""
import ctypes
import os

from ._build import LIB as LIB_PATH

# bst_dtype
F16, BF16, E4M3, S8, F32, S32 = 0, 1, 2, 3, 4, 5
# bst_layout
ROW_MAJOR, COL_MAJOR = 0, 1
# bst_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(7)

EXPORTED = ["bst_gemm", "bst_gemm_batched", "bst_gemm_grouped", "bst_gemm_grouped_quant_per_token",
            "bst_gemm_grouped_quant_per_token_workspace_size", "bst_gemm_grouped_slice_k",
            "bst_gemm_grouped_slice_k_workspace_size", "bst_gemm_grouped_slice_k_quant_per_token",
            "bst_gemm_grouped_slice_k_quant_per_token_workspace_size", "bst_gemm_quant_per_token",
            "bst_gemm_quant_per_token_noalloc", "bst_gemm_quant_per_token_workspace_size", "bst_swizzle_map",
            "bst_swizzle_map_grouped", "bst_check_async", "bst_status_string", "bst_set_wait_timeout_ns",
            "bst_wait_check"]
# BST_NOALLOC_SCRATCH_BYTES: the scratch limit of gemm_quant_per_token_noalloc
NOALLOC_SCRATCH_BYTES = 32 << 20


class BstError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class Sched(ctypes.Structure):
    """bst_sched."""
    _fields_ = [("swizzle_offset", ctypes.c_uint32), ("swizzle_direction", ctypes.c_uint32),
                ("tile_n", ctypes.c_uint32), ("tile_m", ctypes.c_uint32), ("num_ctas", ctypes.c_uint32),
                ("split_k", ctypes.c_uint32),
                ("trace", ctypes.c_void_p), ("timeline", ctypes.c_void_p),
                ("shuffle_k", ctypes.c_uint32), ("dynamic", ctypes.c_uint32)]


def sched(swizzle_offset=1, swizzle_direction=0, tile_n=0, num_ctas=0, trace=None, timeline=None, tile_m=0,
          split_k=0, shuffle_k=0, dynamic=0):
    return Sched(swizzle_offset, swizzle_direction, tile_n, tile_m, num_ctas, split_k, _ptr(trace), _ptr(timeline),
                 shuffle_k, dynamic)


_lib = None

_i64, _u32, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
_SIGS = {
    "bst_gemm": [_i64, _i64, _i64, _vp, _i32, _i32, _i64, _vp, _i32, _i32, _i64, _vp, _i32, _i64, _vp, _vp,
                 ctypes.POINTER(Sched), _vp],
    "bst_gemm_batched": [_i64, _i64, _i64, _vp, _i32, _i32, _i64, _i64, _vp, _i32, _i32, _i64, _i64, _vp, _i32,
                         _i64, _i64, _i64, ctypes.POINTER(Sched), _vp],
    "bst_gemm_grouped": [_i32, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i32, _i64, _i64, _vp, _i64, _i32, _i32,
                         ctypes.POINTER(Sched), _vp],
    "bst_gemm_quant_per_token_workspace_size": [_i64, _i64, _i64],
    "bst_gemm_quant_per_token": [_i64, _i64, _i64, _vp, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _sz,
                                 ctypes.POINTER(Sched), _vp],
    "bst_gemm_grouped_quant_per_token_workspace_size": [_i32, _i64, _i64, _i64],
    "bst_gemm_grouped_quant_per_token": [_i32, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i32, _i64, _i64, _vp, _vp,
                                         _i64, _vp, _i64, _vp, _vp, _sz, ctypes.POINTER(Sched), _vp],
    "bst_gemm_grouped_slice_k_workspace_size": [_i32],
    "bst_gemm_grouped_slice_k": [_i32, _vp, _i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _i64, _i64,
                                 _i32, _i32, _vp, _sz, ctypes.POINTER(Sched), _vp],
    "bst_gemm_grouped_slice_k_quant_per_token_workspace_size": [_i32, _i64, _i64, _i64],
    "bst_gemm_grouped_slice_k_quant_per_token": [_i32, _vp, _i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64,
                                                 _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _sz,
                                                 ctypes.POINTER(Sched), _vp],
    "bst_gemm_quant_per_token_noalloc": [_i64, _i64, _i64, _vp, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i64, _vp,
                                         ctypes.POINTER(Sched), _vp],
    "bst_swizzle_map": [_u32, _u32, _u32, _u32, _u32, ctypes.POINTER(Sched), _vp, _vp],
    "bst_swizzle_map_grouped": [_i32, _vp, _u32, _u32, _u32, ctypes.POINTER(Sched), _vp, _u32, _vp],
    "bst_check_async": [_vp],
    "bst_status_string": [_i32],
    "bst_set_wait_timeout_ns": [ctypes.c_uint64],
    "bst_wait_check": [ctypes.c_uint64, _i32, _vp],
}


def lib():
    """The loaded libbst.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libbst.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.bst_gemm_quant_per_token_workspace_size.restype = ctypes.c_size_t
        L.bst_gemm_grouped_quant_per_token_workspace_size.restype = ctypes.c_size_t
        L.bst_gemm_grouped_slice_k_workspace_size.restype = ctypes.c_size_t
        L.bst_gemm_grouped_slice_k_quant_per_token_workspace_size.restype = ctypes.c_size_t
        L.bst_status_string.restype = ctypes.c_char_p
        L.bst_set_wait_timeout_ns.restype = None
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _sched(s):
    return None if s is None else ctypes.byref(s)


def _check(status, where):
    if status != OK:
        raise BstError(status, where)


def status_string(status):
    return lib().bst_status_string(status).decode()


def gemm(M, N, K, A, a_type, a_layout, lda, B, b_type, b_layout, ldb, C, c_type, ldc,
         scale_a=None, scale_b=None, sched=None, stream=None):
    _check(lib().bst_gemm(M, N, K, _ptr(A), a_type, a_layout, lda, _ptr(B), b_type, b_layout, ldb,
                          _ptr(C), c_type, ldc, _ptr(scale_a), _ptr(scale_b), _sched(sched), _stream(stream)),
           "bst_gemm")


def gemm_batched(M, N, K, A, a_type, a_layout, lda, stride_a, B, b_type, b_layout, ldb, stride_b,
                 C, c_type, ldc, stride_c, batch, sched=None, stream=None):
    _check(lib().bst_gemm_batched(M, N, K, _ptr(A), a_type, a_layout, lda, stride_a, _ptr(B), b_type, b_layout,
                                  ldb, stride_b, _ptr(C), c_type, ldc, stride_c, batch, _sched(sched),
                                  _stream(stream)), "bst_gemm_batched")


def gemm_grouped(G, group_m, total_m, N, K, A, lda, B, b_layout, ldb, stride_b, C, ldc, ab_type, c_type,
                 sched=None, stream=None):
    _check(lib().bst_gemm_grouped(G, _ptr(group_m), total_m, N, K, _ptr(A), lda, _ptr(B), b_layout, ldb, stride_b,
                                  _ptr(C), ldc, ab_type, c_type, _sched(sched), _stream(stream)), "bst_gemm_grouped")


def gemm_quant_per_token_workspace_size(M, N, K):
    return lib().bst_gemm_quant_per_token_workspace_size(M, N, K)


def gemm_quant_per_token(M, N, K, A, lda, B, b_layout, ldb, scale_a, scale_b, C, ldc, acc_out,
                         workspace, workspace_bytes, sched=None, stream=None):
    _check(lib().bst_gemm_quant_per_token(M, N, K, _ptr(A), lda, _ptr(B), b_layout, ldb, _ptr(scale_a),
                                          _ptr(scale_b), _ptr(C), ldc, _ptr(acc_out), _ptr(workspace),
                                          workspace_bytes, _sched(sched), _stream(stream)),
           "bst_gemm_quant_per_token")


def gemm_grouped_quant_per_token_workspace_size(G, total_m, N, K):
    return lib().bst_gemm_grouped_quant_per_token_workspace_size(G, total_m, N, K)


def gemm_grouped_quant_per_token(G, group_m, total_m, N, K, A, lda, B, b_layout, ldb, stride_b, scale_a, scale_b,
                                 stride_sb, C, ldc, acc_out, workspace, workspace_bytes, sched=None, stream=None):
    _check(lib().bst_gemm_grouped_quant_per_token(G, _ptr(group_m), total_m, N, K, _ptr(A), lda, _ptr(B), b_layout,
                                                  ldb, stride_b, _ptr(scale_a), _ptr(scale_b), stride_sb, _ptr(C),
                                                  ldc, _ptr(acc_out), _ptr(workspace), workspace_bytes,
                                                  _sched(sched), _stream(stream)),
           "bst_gemm_grouped_quant_per_token")


def gemm_grouped_slice_k_workspace_size(G):
    return lib().bst_gemm_grouped_slice_k_workspace_size(G)


def gemm_grouped_slice_k(G, group_k, M, N, total_k, A, a_layout, lda, B, b_layout, ldb, C, ldc, stride_c, ab_type,
                         c_type, workspace, workspace_bytes, sched=None, stream=None):
    _check(lib().bst_gemm_grouped_slice_k(G, _ptr(group_k), M, N, total_k, _ptr(A), a_layout, lda, _ptr(B), b_layout,
                                          ldb, _ptr(C), ldc, stride_c, ab_type, c_type, _ptr(workspace),
                                          workspace_bytes, _sched(sched), _stream(stream)),
           "bst_gemm_grouped_slice_k")


def gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, total_k):
    return lib().bst_gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, total_k)


def gemm_grouped_slice_k_quant_per_token(G, group_k, M, N, total_k, A, a_layout, lda, B, b_layout, ldb, scale_a,
                                         stride_sa, scale_b, stride_sb, C, ldc, stride_c, acc_out, workspace,
                                         workspace_bytes, sched=None, stream=None):
    _check(lib().bst_gemm_grouped_slice_k_quant_per_token(G, _ptr(group_k), M, N, total_k, _ptr(A), a_layout, lda,
                                                          _ptr(B), b_layout, ldb, _ptr(scale_a), stride_sa,
                                                          _ptr(scale_b), stride_sb, _ptr(C), ldc, stride_c,
                                                          _ptr(acc_out), _ptr(workspace), workspace_bytes,
                                                          _sched(sched), _stream(stream)),
           "bst_gemm_grouped_slice_k_quant_per_token")


def gemm_quant_per_token_noalloc(M, N, K, A, lda, B, b_layout, ldb, scale_a, scale_b, C, ldc, acc_out,
                                 sched=None, stream=None):
    """gemm_quant_per_token without a workspace argument: the library's own
    fixed scratch of NOALLOC_SCRATCH_BYTES is used and nothing is allocated.
    Problems needing more scratch raise BstError(ERR_UNSUPPORTED)."""
    status = lib().bst_gemm_quant_per_token_noalloc(M, N, K, _ptr(A), lda, _ptr(B), b_layout, ldb, _ptr(scale_a),
                                                    _ptr(scale_b), _ptr(C), ldc, _ptr(acc_out), _sched(sched),
                                                    _stream(stream))
    where = "bst_gemm_quant_per_token_noalloc"
    need = gemm_quant_per_token_workspace_size(M, N, K)
    if status == ERR_UNSUPPORTED and need > NOALLOC_SCRATCH_BYTES:
        where += " (needs %d bytes of scratch, limit %d)" % (need, NOALLOC_SCRATCH_BYTES)
    _check(status, where)


def swizzle_map(M, N, tile_m, tile_n, batch, sched, out, stream=None):
    _check(lib().bst_swizzle_map(M, N, tile_m, tile_n, batch, _sched(sched), _ptr(out), _stream(stream)),
           "bst_swizzle_map")


def swizzle_map_grouped(G, group_m, N, tile_m, tile_n, sched, out, max_tasks, stream=None):
    _check(lib().bst_swizzle_map_grouped(G, _ptr(group_m), N, tile_m, tile_n, _sched(sched), _ptr(out),
                                         max_tasks, _stream(stream)), "bst_swizzle_map_grouped")


def check_async(stream=None):
    """Synchronises the stream and raises if a kernel reported a device-side
    failure since the last check."""
    _check(lib().bst_check_async(_stream(stream)), "bst_check_async")


def set_wait_timeout_ns(ns):
    lib().bst_set_wait_timeout_ns(ns)


def wait_check(timeout_ns, arrive, stream=None):
    """Launches the bounded-wait self-check (bst_wait_check); the result is
    reported by the next check_async."""
    _check(lib().bst_wait_check(timeout_ns, 1 if arrive else 0, _stream(stream)), "bst_wait_check")
