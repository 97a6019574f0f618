"""CPU checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every function include/bst.h declares, and rejects invalid
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bst.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bst.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bst_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["bst_gemm", "bst_gemm_batched", "bst_gemm_grouped", "bst_gemm_quant_per_token",
                 "bst_swizzle_map", "bst_swizzle_map_grouped", "bst_check_async", "bst_status_string"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(bst.EXPORTED) == declared_functions()


def test_status_strings(lib):
    for s in range(7):
        assert bst.status_string(s) and bst.status_string(s) != "unknown status"


def test_workspace_size(lib):
    # A [M, K8] and B [max(N*K8, K*N8)] in bf16, each rounded to 256 bytes
    assert bst.gemm_quant_per_token_workspace_size(8192, 8192, 8192) == 2 * 8192 * 8192 * 2
    assert bst.gemm_quant_per_token_workspace_size(3, 5, 7) == 256 + 256
    assert bst.gemm_quant_per_token_workspace_size(-1, 5, 7) == 0


def _gemm_status(lib, **kw):
    args = dict(M=16, N=16, K=16, A=1 << 20, at=bst.F16, al=bst.ROW_MAJOR, lda=16, B=1 << 20, bt=bst.F16,
                bl=bst.ROW_MAJOR, ldb=16, C=1 << 20, ct=bst.F16, ldc=16, sa=None, sb=None, sched=None)
    args.update(kw)
    s = args["sched"]
    return lib.bst_gemm(args["M"], args["N"], args["K"], args["A"], args["at"], args["al"], args["lda"],
                        args["B"], args["bt"], args["bl"], args["ldb"], args["C"], args["ct"], args["ldc"],
                        args["sa"], args["sb"], ctypes.byref(s) if s is not None else None, None)


def test_argument_errors_need_no_device(lib):
    # every case below is rejected before any CUDA call
    assert _gemm_status(lib, M=-1) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, K=-5) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, at=bst.F16, bt=bst.BF16) == bst.ERR_UNSUPPORTED
    assert _gemm_status(lib, ct=bst.S8) == bst.ERR_UNSUPPORTED
    assert _gemm_status(lib, ldc=15) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, lda=8) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, al=7) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, sched=bst.sched(0, 0)) == bst.ERR_INVALID_ARG      # SwizzleOffset 0
    assert _gemm_status(lib, sched=bst.sched(1, 2)) == bst.ERR_INVALID_ARG      # direction 2
    assert _gemm_status(lib, sched=bst.sched(1, 0, tile_n=96)) == bst.ERR_INVALID_ARG
    assert _gemm_status(lib, sa=1 << 20) == bst.ERR_INVALID_ARG                 # scales without e4m3
    assert _gemm_status(lib, at=bst.E4M3, bt=bst.E4M3, al=bst.COL_MAJOR) == bst.ERR_UNSUPPORTED
    assert _gemm_status(lib, at=bst.E4M3, bt=bst.E4M3, bl=bst.COL_MAJOR, K=96) == bst.ERR_UNSUPPORTED
    assert _gemm_status(lib, C=None) == bst.ERR_INVALID_ARG
    # empty outputs are a no-op and need no device either
    assert _gemm_status(lib, M=0, A=None, B=None, C=None) == bst.OK
    assert lib.bst_gemm_grouped(0, None, 0, 1, 1, None, 1, None, 0, 1, 0, None, 1, bst.BF16, bst.BF16,
                                None, None) == bst.ERR_INVALID_ARG
    assert lib.bst_gemm_grouped(2000, 1, 10, 1, 1, 1, 1, 1, 0, 1, 0, 1, 1, bst.BF16, bst.BF16,
                                None, None) == bst.ERR_INVALID_ARG
    assert lib.bst_swizzle_map(10, 10, 0, 4, 1, None, 1, None) == bst.ERR_INVALID_ARG
    assert lib.bst_swizzle_map(1 << 31, 1 << 31, 1, 1, 1, None, 1, None) == bst.ERR_INVALID_ARG
    # the bounded-wait self-check: its limit is checked before any device work
    assert lib.bst_wait_check(0, 0, None) == bst.ERR_INVALID_ARG
    assert lib.bst_wait_check(10_000_000_001, 1, None) == bst.ERR_INVALID_ARG


def test_noalloc_rejects_oversize_without_a_device(lib):
    # 4096^3 needs 64 MiB of scratch, past the 32 MiB array: rejected before any CUDA call
    assert bst.gemm_quant_per_token_workspace_size(4096, 4096, 4096) > bst.NOALLOC_SCRATCH_BYTES
    s = lib.bst_gemm_quant_per_token_noalloc(4096, 4096, 4096, 1 << 20, 4096, 1 << 20, bst.COL_MAJOR, 4096,
                                             1 << 20, 1 << 20, 1 << 20, 4096, None, None, None)
    assert s == bst.ERR_UNSUPPORTED
    assert lib.bst_gemm_quant_per_token_noalloc(-1, 4, 4, None, 4, None, bst.COL_MAJOR, 4, None, None, None, 4,
                                                None, None, None) == bst.ERR_INVALID_ARG


def test_noalloc_limit_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define BST_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == bst.NOALLOC_SCRATCH_BYTES
