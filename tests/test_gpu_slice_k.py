"""GPU parity of grouped slice-K (bf16/fp16 and int8 with per-token
dequant) against the CPU oracle: ragged and empty groups, every operand
layout, tails in M and N, the task trace against the oracle scheduler, size
errors the kernel must report, and every element of the full workloads."""
import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from oracle import gemm as og, swizzle as osw
from tests.gpu_util import FRO_MX, assert_close_f16, assert_close_fro, canary_intact, decode_out, dev, empty_bytes, host

pytestmark = pytest.mark.gpu
CANARY = 256


def _pad8(x):
    return -(-x // 8) * 8


def store_a(a, row_major, esize):
    """Logical A [M, K] -> (storage with a padded pitch, lda).  Row-major keeps
    K contiguous; column-major stores A^T ([K, M], M contiguous)."""
    src = a if row_major else a.T
    ld = max(8, _pad8(src.shape[1])) if esize == 2 else max(16, -(-src.shape[1] // 16) * 16)
    buf = np.zeros((src.shape[0], ld), dtype=src.dtype)
    buf[:, :src.shape[1]] = src
    return buf, ld


def store_b(b, row_major, esize):
    """Logical B [K, N] -> storage: row-major [K, N] or column-major [N, K]."""
    return store_a(b, row_major, esize)


def run_slice_k(a_bits, b_bits, gk, a_row, b_row, ab="bf16", out="bf16", sched=None, gdev=None, total_k=None):
    M, K = a_bits.shape
    N = b_bits.shape[1]
    G = len(gk)
    total_k = K if total_k is None else total_k
    A, lda = store_a(a_bits, a_row, 2)
    B, ldb = store_b(b_bits, b_row, 2)
    gdev = torch.tensor(gk, dtype=torch.int32, device="cuda") if gdev is None else gdev
    ob = 4 if out == "f32" else 2
    cbuf, C = empty_bytes(G * M * N * ob, CANARY)
    ws_bytes = bst.gemm_grouped_slice_k_workspace_size(G)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    types = {"bf16": bst.BF16, "f16": bst.F16, "f32": bst.F32}
    bst.gemm_grouped_slice_k(G, gdev, M, N, total_k, dev(A), bst.ROW_MAJOR if a_row else bst.COL_MAJOR, lda,
                             dev(B), bst.ROW_MAJOR if b_row else bst.COL_MAJOR, ldb, C, N, M * N, types[ab],
                             types[out], ws, ws_bytes, sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    raw = host(C, np.uint8).view(np.float32 if out == "f32" else np.uint16).reshape(G, M, N)
    return decode_out(raw.copy(), out)


def oracle_slice_k(a_bits, b_bits, gk, ab, out):
    return decode_out(og.gemm_grouped_slice_k(og.decode(a_bits, ab), og.decode(b_bits, ab), gk, out), out)


def check_groups(got, ref, gk):
    for g, kg in enumerate(gk):
        if kg == 0:
            assert not got[g].any(), "empty group %d must be zero" % g
        else:
            assert_close_f16(got[g], ref[g])


def make(gk, M, N, ab="bf16", seed=0):
    w = wl.grouped_slice_k_bf16(group_k=gk, M=M, N=N, seed=seed) if ab == "bf16" else None
    if w is not None:
        return np.ascontiguousarray(w["x"].T), w["dy"]          # logical A [M, K], B [K, N]
    g = wl._gen(seed)
    K = sum(gk)
    return wl.normal16((M, K), 1.0, ab, g), wl.normal16((K, N), 1.0, ab, g)


@pytest.mark.parametrize("gk", [[1, 0, 63, 64, 65, 300], [0, 0, 5], [700], [2] * 12, [0, 129, 0]])
def test_slice_k_mn_major_ragged(gk):
    """The weight-gradient layout (A^T and B both stored [K, rows]): any
    group size works, including 1, empty and sub-k-block groups."""
    a, b = make(gk, 300, 520, seed=len(gk))
    got = run_slice_k(a, b, gk, a_row=False, b_row=True)
    check_groups(got, oracle_slice_k(a, b, gk, "bf16", "bf16"), gk)


@pytest.mark.parametrize("a_row,b_row", [(True, False), (True, True), (False, False)])
def test_slice_k_layouts(a_row, b_row):
    """K-contiguous operands need each group to start on a 16-byte boundary:
    sizes that are multiples of 8 (the last may be ragged)."""
    gk = [8, 0, 136, 64, 200, 13]
    a, b = make(gk, 260, 300, seed=3)
    got = run_slice_k(a, b, gk, a_row, b_row)
    check_groups(got, oracle_slice_k(a, b, gk, "bf16", "bf16"), gk)


def test_slice_k_f16_to_f32_and_tile_128():
    gk = [40, 0, 250, 9]
    a, b = make(gk, 130, 200, ab="f16", seed=4)
    ref = oracle_slice_k(a, b, gk, "f16", "f32")
    check_groups(run_slice_k(a, b, gk, False, True, ab="f16", out="f32"), ref, gk)
    check_groups(run_slice_k(a, b, gk, False, True, ab="f16", out="f32", sched=bst.sched(1, 0, tile_n=128)), ref, gk)


@pytest.mark.parametrize("S,d", [(1, 0), (2, 1), (3, 0)])
def test_slice_k_trace_is_the_batched_map(S, d):
    """Tasks are numbered group-major; each group is one batch of the
    scheduler on the M x N tile grid."""
    gk = [70, 0, 130]
    M, N = 600, 700
    a, b = make(gk, M, N, seed=5)
    tiles = 3 * (-(-M // 256)) * (-(-N // 256))
    trace = torch.full((tiles * 5,), -1, dtype=torch.int32, device="cuda")
    got = run_slice_k(a, b, gk, False, True, sched=bst.sched(S, d, tile_n=256, trace=trace))
    check_groups(got, oracle_slice_k(a, b, gk, "bf16", "bf16"), gk)
    want = np.array(osw.swizzle_map(M, N, 256, 256, S, d, batch=3), dtype=np.uint32)
    assert np.array_equal(trace.cpu().numpy().view(np.uint32).reshape(-1, 5), want)


@pytest.mark.parametrize("gk,total_k,a_row", [([5, 11], 16, True), ([10, 20], 24, False), ([8, -1, 9], 17, False)])
def test_slice_k_bad_sizes_reported(gk, total_k, a_row):
    """A K-contiguous group starting off a 16-byte boundary, sizes past the
    operands' K, a negative size: nothing is written, BST_ERR_DEVICE."""
    M, N = 64, 64
    g = wl._gen(6)
    a = wl.normal16((M, total_k), 1.0, "bf16", g)
    b = wl.normal16((total_k, N), 1.0, "bf16", g)
    gdev = torch.tensor(gk, dtype=torch.int32, device="cuda")
    with pytest.raises(bst.BstError) as e:
        run_slice_k(a, b, [0] * len(gk), a_row, True, gdev=gdev)
    assert e.value.status == bst.ERR_DEVICE
    bst.check_async()


def test_slice_k_zero_total_k_zeroes_outputs():
    a = np.zeros((40, 0), np.uint16)
    b = np.zeros((0, 24), np.uint16)
    got = run_slice_k(a, b, [0, 0, 0], True, True)
    assert not got.any()


def test_slice_k_full_workload():
    """G = 8 groups summing to 8192 tokens, M = N = 4096 (the bench
    workload, called as the bench calls it): every element of every C_g."""
    w = wl.grouped_slice_k_bf16()
    gk, M, N = w["group_k"], w["M"], w["N"]
    G = len(gk)
    X, DY = dev(w["x"]), dev(w["dy"])
    gdev = torch.tensor(gk, dtype=torch.int32, device="cuda")
    C = torch.empty(G * M * N, dtype=torch.int16, device="cuda")
    ws_bytes = bst.gemm_grouped_slice_k_workspace_size(G)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bst.gemm_grouped_slice_k(G, gdev, M, N, sum(gk), X, bst.COL_MAJOR, M, DY, bst.ROW_MAJOR, N, C, N, M * N,
                             bst.BF16, bst.BF16, ws, ws_bytes, sched=bst.sched(1, 0))
    bst.check_async()
    out = decode_out(C.cpu().numpy().view(np.uint16).reshape(G, M, N), "bf16")
    xa = og.decode(w["x"], "bf16")
    dy = og.decode(w["dy"], "bf16")
    ref = og.gemm_grouped_slice_k(np.ascontiguousarray(xa.T), dy, gk, "bf16")
    check_groups(out, decode_out(ref, "bf16"), gk)


# ------------------------------------------------ int8, per-token dequant --

def run_slice_k_int8(w, a_row, b_row, sched=None, share_sa=False):
    gk, M, N = w["group_k"], w["M"], w["N"]
    G = len(gk)
    K = sum(gk)
    A, lda = store_a(w["a"], a_row, 1)
    B, ldb = store_b(w["b"], b_row, 1)
    sa = w["sa"][:1] if share_sa else w["sa"]
    gdev = torch.tensor(gk, dtype=torch.int32, device="cuda")
    cbuf, C = empty_bytes(G * M * N * 2, CANARY)
    abuf, ACC = empty_bytes(G * M * N * 4, CANARY)
    ws_bytes = bst.gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bst.gemm_grouped_slice_k_quant_per_token(G, gdev, M, N, K, dev(A), bst.ROW_MAJOR if a_row else bst.COL_MAJOR,
                                             lda, dev(B), bst.ROW_MAJOR if b_row else bst.COL_MAJOR, ldb, dev(sa),
                                             0 if share_sa else M, dev(w["sb"]), N, C, N, M * N, ACC, ws, ws_bytes,
                                             sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY) and canary_intact(abuf, CANARY)
    out = decode_out(host(C, np.uint16).reshape(G, M, N).copy(), "bf16")
    return out, host(ACC, np.int32).reshape(G, M, N).copy()


@pytest.mark.parametrize("a_row,b_row", [(False, True), (True, False)])
@pytest.mark.parametrize("share_sa", [False, True])
def test_slice_k_int8_small(a_row, b_row, share_sa):
    """Exact int32 accumulators; a group of 2100 K spans three exact
    K-chunks; empty groups give zeros."""
    gk = [8, 0, 2104, 64, 24] if a_row else [3, 0, 2100, 65, 17]
    w = wl.grouped_slice_k_int8(group_k=gk, M=300, N=280, seed=8)
    out, acc = run_slice_k_int8(w, a_row, b_row, share_sa=share_sa)
    sa = np.repeat(w["sa"][:1], len(gk), axis=0) if share_sa else w["sa"]
    racc, rout = og.gemm_grouped_slice_k_quant_per_token(w["a"], w["b"], gk, sa, w["sb"])
    assert np.array_equal(acc, racc)
    rout = decode_out(rout, "bf16")
    for g, kg in enumerate(gk):
        if kg:
            assert_close_fro(out[g], rout[g], FRO_MX)
        else:
            assert not out[g].any()


def test_slice_k_int8_full_workload_without_acc_out():
    """The int8 slice-K bench workload (G = 8, K sizes over 8192 tokens,
    M = N = 4096, A^T [K, M] and B [K, N]) called as the bench calls it
    (acc_out = NULL): every bf16 output of every group within the dequant
    tolerance of the oracle."""
    w = wl.grouped_slice_k_int8()
    gk, M, N = w["group_k"], w["M"], w["N"]
    G, K = len(gk), sum(gk)
    A = dev(np.ascontiguousarray(w["a"].T))
    B = dev(w["b"])
    gdev = torch.tensor(gk, dtype=torch.int32, device="cuda")
    cbuf, C = empty_bytes(G * M * N * 2, CANARY)
    ws_bytes = bst.gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bst.gemm_grouped_slice_k_quant_per_token(G, gdev, M, N, K, A, bst.COL_MAJOR, M, B, bst.ROW_MAJOR, N,
                                             dev(w["sa"]), M, dev(w["sb"]), N, C, N, M * N, None, ws, ws_bytes,
                                             sched=bst.sched(1, 0))
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    out = decode_out(host(C, np.uint16).reshape(G, M, N).copy(), "bf16")
    _, rout = og.gemm_grouped_slice_k_quant_per_token(w["a"], w["b"], gk, w["sa"], w["sb"])
    rout = decode_out(rout, "bf16")
    for g, kg in enumerate(gk):
        if kg:
            assert_close_fro(out[g], rout[g], FRO_MX)
        else:
            assert not out[g].any()
