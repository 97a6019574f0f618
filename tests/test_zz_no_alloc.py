"""GPU check of bst_gemm_quant_per_token_noalloc, the int8 per-token GEMM
entry point that takes its scratch from the library's fixed array instead of
a caller workspace.  Its results must equal those of
bst_gemm_quant_per_token on the same inputs bit for bit (the same kernels run
on the same bytes: exact int32 accumulators and identical bf16 outputs, which
are also within the dequant tolerance of each other), on two calls issued
back to back, and a call must leave the device's free memory unchanged."""
import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from tests.gpu_util import FRO_MX, assert_close_fro, canary_intact, decode_out, dev, empty_bytes, host

pytestmark = pytest.mark.gpu
CANARY = 256


def _buffers(M, N):
    cbuf, C = empty_bytes(M * N * 2, CANARY)
    abuf, ACC = empty_bytes(M * N * 4, CANARY)
    return cbuf, C, abuf, ACC


def _results(M, N, C, ACC):
    out = decode_out(host(C, np.uint16).reshape(M, N).copy(), "bf16")
    acc = host(ACC, np.int32).reshape(M, N).copy()
    return out, acc


def _with_workspace(w, b_col):
    """The existing entry point, with a caller-owned workspace."""
    M, N, K = w["M"], w["N"], w["K"]
    Bst = w["b"] if b_col else np.ascontiguousarray(w["b"].T)
    _, C, _, ACC = _buffers(M, N)
    ws_bytes = bst.gemm_quant_per_token_workspace_size(M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bst.gemm_quant_per_token(M, N, K, dev(w["a"]), K, dev(Bst), bst.COL_MAJOR if b_col else bst.ROW_MAJOR,
                             K if b_col else N, dev(w["sa"]), dev(w["sb"]), C, N, ACC, ws, ws_bytes)
    bst.check_async()
    return _results(M, N, C, ACC)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    cases = [(wl.int8_per_token(1000, 768, 2100, seed=11), True),
             (wl.int8_per_token(300, 520, 1030, seed=12), False)]
    want = [_with_workspace(w, b_col) for w, b_col in cases]
    torch.cuda.synchronize()
    # both calls enqueued back to back on one stream, no host sync between
    held = []
    for w, b_col in cases:
        M, N, K = w["M"], w["N"], w["K"]
        assert bst.gemm_quant_per_token_workspace_size(M, N, K) <= bst.NOALLOC_SCRATCH_BYTES
        Bst = w["b"] if b_col else np.ascontiguousarray(w["b"].T)
        A, B, SA, SB = dev(w["a"]), dev(Bst), dev(w["sa"]), dev(w["sb"])
        cbuf, C, abuf, ACC = _buffers(M, N)
        bst.gemm_quant_per_token_noalloc(M, N, K, A, K, B, bst.COL_MAJOR if b_col else bst.ROW_MAJOR,
                                         K if b_col else N, SA, SB, C, N, ACC)
        held.append((M, N, cbuf, C, abuf, ACC, A, B, SA, SB))
    bst.check_async()
    for (M, N, cbuf, C, abuf, ACC, *_), (wout, wacc) in zip(held, want):
        assert canary_intact(cbuf, CANARY) and canary_intact(abuf, CANARY)
        out, acc = _results(M, N, C, ACC)
        assert np.array_equal(acc, wacc)
        assert np.array_equal(out.view(np.uint64), wout.view(np.uint64))
        assert_close_fro(out, wout, FRO_MX)


def test_noalloc_call_leaves_free_device_memory_unchanged():
    """After one warm-up call (which only looks up the scratch array's
    address), a further call allocates no device memory: the free memory the
    driver reports is the same before and after it."""
    w = wl.int8_per_token(512, 384, 1024, seed=13)
    M, N, K = w["M"], w["N"], w["K"]
    A, B, SA, SB = dev(w["a"]), dev(w["b"]), dev(w["sa"]), dev(w["sb"])
    _, C, _, ACC = _buffers(M, N)
    bst.gemm_quant_per_token_noalloc(M, N, K, A, K, B, bst.COL_MAJOR, K, SA, SB, C, N, ACC)
    bst.check_async()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    bst.gemm_quant_per_token_noalloc(M, N, K, A, K, B, bst.COL_MAJOR, K, SA, SB, C, N, ACC)
    bst.check_async()
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_noalloc_rejects_problems_past_the_scratch_limit():
    M = N = K = 4096             # needs 64 MiB of scratch
    assert bst.gemm_quant_per_token_workspace_size(M, N, K) > bst.NOALLOC_SCRATCH_BYTES
    with pytest.raises(bst.BstError) as e:
        bst.gemm_quant_per_token_noalloc(M, N, K, 1 << 20, K, 1 << 20, bst.COL_MAJOR, K, 1 << 20, 1 << 20,
                                         1 << 20, N, None)
    assert e.value.status == bst.ERR_UNSUPPORTED
    assert "limit" in str(e.value)
