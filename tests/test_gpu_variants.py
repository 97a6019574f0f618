"""GPU parity of the grouped slice-M, MXFP8 and int8 per-token-dequant paths
against the CPU oracle, at small ragged sizes and at the full workload sizes
(full sizes compare every output element)."""
import functools

import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from oracle import formats, gemm as og, swizzle as osw
from tests.gpu_util import (FRO_MX, assert_close_f16, assert_close_fro, assert_special_equal, canary_intact,
                            decode_out, dev, empty_bytes, host)

pytestmark = pytest.mark.gpu
CANARY = 256


# ------------------------------------------------------------- grouped -----

def run_grouped(w, sched=None, b_col_major=False, out="bf16"):
    gm, N, K = w["group_m"], w["N"], w["K"]
    G = len(gm)
    total = sum(gm)
    X = dev(w["x"])
    W = w["w"]
    if b_col_major:                                   # store each B_g as [N, K]
        W = np.ascontiguousarray(np.transpose(W, (0, 2, 1)))
    Wd = dev(W)
    gdev = torch.tensor(gm, dtype=torch.int32, device="cuda")
    ob = 4 if out == "f32" else 2
    cbuf, C = empty_bytes(max(total, 1) * N * ob, CANARY)
    bst.gemm_grouped(G, gdev, total, N, K, X, K, Wd, bst.COL_MAJOR if b_col_major else bst.ROW_MAJOR,
                     K if b_col_major else N, K * N, C, N, bst.BF16, {"bf16": bst.BF16, "f32": bst.F32}[out],
                     sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    raw = host(C, np.uint8).view(np.float32 if out == "f32" else np.uint16).reshape(-1, N)[:total]
    return decode_out(raw.copy(), out)


@pytest.mark.parametrize("gm", [[3, 0, 130, 1, 0, 257], [0, 0, 64], [200], [1] * 17, [300, 0, 513]])
@pytest.mark.parametrize("bcol", [False, True])
def test_grouped_small(gm, bcol):
    w = wl.grouped_bf16(group_m=gm, N=200, K=136, seed=len(gm))
    total = sum(gm)
    for S, d, tm, tn in [(1, 0, 128, 128), (2, 1, 128, 64), (3, 0, 128, 256), (1, 1, 256, 256), (2, 0, 256, 128)]:
        G = len(gm)
        cap = (-(-total // tm) + G) * -(-200 // tn)
        trace = torch.full((cap * 5,), -1, dtype=torch.int32, device="cuda")
        got = run_grouped(w, bst.sched(S, d, tile_n=tn, tile_m=tm, trace=trace), b_col_major=bcol)
        ref = decode_out(og.gemm_grouped(og.decode(w["x"], "bf16"), og.decode(w["w"], "bf16"), gm, "bf16"), "bf16")
        assert_close_f16(got, ref)
        want = np.array(osw.grouped_swizzle_map(gm, 200, tm, tn, S, d), dtype=np.uint32).reshape(-1, 5)
        tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)[:len(want)]
        assert np.array_equal(tr, want)


def test_grouped_inconsistent_sizes_reported():
    w = wl.grouped_bf16(group_m=[100, 100], N=64, K=64, seed=1)
    gdev = torch.tensor([100, 200], dtype=torch.int32, device="cuda")     # sums past total_m = 200
    X, Wd = dev(w["x"]), dev(w["w"])
    C = torch.zeros(200 * 64, dtype=torch.int16, device="cuda")
    bst.gemm_grouped(2, gdev, 200, 64, 64, X, 64, Wd, bst.ROW_MAJOR, 64, 64 * 64, C, 64, bst.BF16, bst.BF16)
    with pytest.raises(bst.BstError) as e:
        bst.check_async()
    assert e.value.status == bst.ERR_DEVICE
    bst.check_async()      # the error word was cleared


@functools.lru_cache(maxsize=1)
def _grouped_full_oracle(forced):
    w = wl.grouped_bf16(group_m=None if forced is None else list(forced))
    ref = decode_out(og.gemm_grouped(og.decode(w["x"], "bf16"), og.decode(w["w"], "bf16"), w["group_m"], "bf16"),
                     "bf16")
    return w, ref


@pytest.mark.parametrize("forced", [None, (0, 2048, 0, 1024, 3072, 0, 2048, 0)])
@pytest.mark.parametrize("tm", [0, 128, 256])
def test_grouped_full_workload(forced, tm):
    """G=8 groups summing to 8192 rows, K=N=4096, bf16: every element of the
    output against the oracle (tm 0 is the automatic choice the bench
    times)."""
    w, ref = _grouped_full_oracle(forced)
    for S, d in ([(1, 0), (8, 1)] if tm == 0 else [(1, 0)]):
        got = run_grouped(w, bst.sched(S, d, tile_m=tm))
        assert_close_f16(got, ref)


# --------------------------------------------------------------- MXFP8 -----

def run_mx(w, sched=None, out="bf16"):
    M, N, K = w["M"], w["N"], w["K"]
    A, B, SA, SB = dev(w["a"]), dev(w["b"]), dev(w["sa"]), dev(w["sb"])
    ob = 4 if out == "f32" else 2
    cbuf, C = empty_bytes(M * N * ob, CANARY)
    bst.gemm(M, N, K, A, bst.E4M3, bst.ROW_MAJOR, K, B, bst.E4M3, bst.COL_MAJOR, K, C,
             {"bf16": bst.BF16, "f32": bst.F32}[out], N, scale_a=SA, scale_b=SB, sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    raw = host(C, np.uint8).view(np.float32 if out == "f32" else np.uint16).reshape(M, N)
    return decode_out(raw.copy(), out)


@pytest.mark.parametrize("mnk", [(128, 128, 128), (200, 300, 256), (129, 257, 512), (1, 40, 128)])
@pytest.mark.parametrize("tn", [128, 256])
def test_mxfp8_small(mnk, tn):
    M, N, K = mnk
    w = wl.mxfp8(M, N, K, seed=M + N)
    got = run_mx(w, bst.sched(2, 0, tile_n=tn))
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"]), "bf16")
    assert_close_fro(got, ref, FRO_MX)


def test_mxfp8_unit_scales_and_single_block():
    """All scales 1 except one 32-block of one row of A: checks each scale
    reaches exactly its own rows and K sub-block."""
    M, N, K = 256, 256, 256
    w = wl.mxfp8(M, N, K, seed=3)
    w["sa"][:] = 127
    w["sb"][:] = 127
    w["sa"][37, 5] = 130          # x8 on row 37, K 160..191
    w["sb"][200, 2] = 124         # /8 on column 200, K 64..95
    got = run_mx(w, bst.sched(1, 0, tile_n=128), out="f32")
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"], "f32"), "f32")
    assert_close_fro(got, ref, 1e-5)


@pytest.mark.parametrize("K", [256, 1024])
def test_mxfp8_nan_code_and_nan_scale(K):
    """The NaN encodings of the MX formats: e4m3 S.1111.111 in row 5 of A makes
    output row 5 NaN; the E8M0 scale 0xFF on a 32-element block of column 200
    of B makes output column 200 NaN.  K = 256 runs one-CTA tiles, K = 1024
    the CTA pair.  NaN positions equal the oracle's; the rest is within the
    tolerance."""
    M, N = 256, 256
    w = wl.mxfp8(M, N, K, seed=11)
    w["a"][5, 77] = 0x7F
    w["sb"][200, 3] = 0xFF
    got = run_mx(w, bst.sched(1, 0, tile_n=128))
    # the oracle's operands, summed without BLAS, rounded once by the oracle
    acc = np.einsum("ik,jk->ij", og.mx_dequant_operand(w["a"], w["sa"]), og.mx_dequant_operand(w["b"], w["sb"]))
    ref = decode_out(og.round_out(acc, "bf16"), "bf16")
    assert np.isnan(ref[5]).all() and np.isnan(ref[:, 200]).all() and np.isnan(ref).sum() == M + N - 1
    assert_special_equal(got, ref, FRO_MX)


@pytest.mark.parametrize("tn", [128, 256])
def test_mxfp8_scale_placement_tma_path(tn):
    """K = 1024 (scale rows of 32 bytes: the scale factors arrive by TMA in
    16-byte groups of 4 k-blocks): single bumped codes in different groups and
    sub-blocks reach exactly their own row / column and 32-element block."""
    M, N, K = 300, 300, 1024
    w = wl.mxfp8(M, N, K, seed=4)
    w["sa"][:] = 127
    w["sb"][:] = 127
    w["sa"][37, 13] = 130          # x8 on row 37, K 416..447 (k-block 3, group 0)
    w["sa"][160, 20] = 125         # /4 on row 160, K 640..671 (k-block 5, group 1)
    w["sb"][200, 30] = 124         # /8 on column 200, K 960..991 (k-block 7, group 1)
    w["sb"][299, 1] = 129          # x4 on the last column, K 32..63
    got = run_mx(w, bst.sched(1, 0, tile_n=tn), out="f32")
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"], "f32"), "f32")
    assert_close_fro(got, ref, 1e-5)


@pytest.mark.parametrize("tn,splits", [(256, 2), (128, 2), (128, 4)])
@pytest.mark.parametrize("mnk", [(200, 300, 1024), (129, 257, 512), (300, 520, 384), (1024, 512, 4096)])
def test_mxfp8_split_k(tn, splits, mnk):
    """Split-K over clusters of 2 or 4 CTAs (one 128 x tn tile per cluster,
    partials summed in distributed shared memory).  K = 1024 and 512 take the
    TMA scale path in 4-k-block groups, so some splits get no k-blocks; K = 384
    takes the row-by-row scale path."""
    M, N, K = mnk
    w = wl.mxfp8(M, N, K, seed=M + tn + splits)
    lm, ln = -(-M // 128), -(-N // tn)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_mx(w, bst.sched(2, 1, tile_n=tn, split_k=splits, trace=trace))
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"]), "bf16")
    assert_close_fro(got, ref, FRO_MX)
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 128, tn, 2, 1), dtype=np.uint32))


def test_mxfp8_split_k_f32_out_unit_scales():
    M, N, K = 256, 256, 2048
    w = wl.mxfp8(M, N, K, seed=11)
    w["sa"][:] = 127
    w["sb"][:] = 127
    w["sa"][5, 60] = 129            # second half of K: the other split
    w["sb"][250, 3] = 126           # first half of K
    got = run_mx(w, bst.sched(1, 0, tile_n=256, split_k=2), out="f32")
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"], "f32"), "f32")
    assert_close_fro(got, ref, 1e-5)


@pytest.mark.parametrize("tn", [128, 256])
def test_mxfp8_pair_scale_placement(tn):
    """CTA-pair MXFP8 tiles (256 x tn): each CTA's tensor memory must get the
    scale codes of its own 128 rows of A and of all tn columns of B.  Single
    bumped codes in both CTAs' row halves and in both halves of the columns,
    in different 4-k-block groups, reach exactly their own row / column and
    32-element block."""
    M, N, K = 256, 2 * tn, 1024
    w = wl.mxfp8(M, N, K, seed=5 + tn)
    w["sa"][:] = 127
    w["sb"][:] = 127
    w["sa"][37, 13] = 130          # leader's rows: x8 on row 37, k-block 3
    w["sa"][200, 20] = 125         # peer's rows: /4 on row 200, k-block 5 (second group)
    w["sa"][255, 0] = 128          # last row, first block
    w["sb"][5, 30] = 124           # first half of the first tile's columns
    w["sb"][tn - 1, 1] = 129       # second half of the first tile's columns
    w["sb"][tn + 3, 9] = 126       # the second column tile
    trace = torch.zeros(2 * 5, dtype=torch.int32, device="cuda")
    got = run_mx(w, bst.sched(1, 0, tile_m=256, tile_n=tn, trace=trace), out="f32")
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"], "f32"), "f32")
    assert_close_fro(got, ref, 1e-5)
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 256, tn, 1, 0), dtype=np.uint32))


@pytest.mark.parametrize("tn", [128, 256])
@pytest.mark.parametrize("mnk", [(300, 520, 1024), (129, 257, 3072), (1, 40, 1024), (700, 1000, 2048)])
def test_mxfp8_pair_shapes(tn, mnk):
    """Ragged tails in M and N on CTA-pair tiles, several tiles per pair
    (persistent grid), K of one to three 8-k-block groups."""
    M, N, K = mnk
    w = wl.mxfp8(M, N, K, seed=M + N + tn)
    lm, ln = -(-M // 256), -(-N // tn)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_mx(w, bst.sched(3, 1, tile_m=256, tile_n=tn, num_ctas=4, trace=trace))
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"]), "bf16")
    assert_close_fro(got, ref, FRO_MX)
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 256, tn, 3, 1), dtype=np.uint32))


@pytest.mark.parametrize("K", [384, 512])
def test_mxfp8_pair_needs_whole_code_groups(K):
    """CTA-pair MXFP8 tiles take the scale codes in groups of 8 k-blocks (K a
    multiple of 1024): forcing them with K = 384 or 512 is refused; the
    automatic choice still runs (on one-CTA tiles)."""
    w = wl.mxfp8(256, 256, K, seed=6)
    with pytest.raises(bst.BstError) as e:
        run_mx(w, bst.sched(1, 0, tile_m=256))
    assert e.value.status == bst.ERR_UNSUPPORTED
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"]), "bf16")
    assert_close_fro(run_mx(w, bst.sched(1, 0)), ref, FRO_MX)


def test_mxfp8_full_workload():
    """e4m3 1024x2048x4096 with E8M0 scales 2^U{-4..4} per 32 K."""
    w = wl.mxfp8()
    ref = decode_out(og.gemm_mxfp8(w["a"], w["sa"], w["b"], w["sb"]), "bf16")
    # the automatic choice (CTA pairs), then one-CTA tiles split in two
    for S, d, kw in [(1, 0, {}), (8, 1, {}), (4, 1, dict(tile_m=128, split_k=2))]:
        got = run_mx(w, bst.sched(S, d, **kw))
        assert_close_fro(got, ref, FRO_MX)


# ---------------------------------------------------------------- int8 -----

def run_int8(w, b_col_major=True, sched=None, with_acc=True):
    """One bst_gemm_quant_per_token call; with_acc=False passes acc_out =
    NULL (the call the bench times) and returns acc None."""
    M, N, K = w["M"], w["N"], w["K"]
    Bst = w["b"] if b_col_major else np.ascontiguousarray(w["b"].T)
    A, B = dev(w["a"]), dev(Bst)
    SA, SB = dev(w["sa"]), dev(w["sb"])
    cbuf, C = empty_bytes(M * N * 2, CANARY)
    abuf, ACC = empty_bytes(M * N * 4, CANARY) if with_acc else (None, None)
    ws_bytes = bst.gemm_quant_per_token_workspace_size(M, N, K)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    bst.gemm_quant_per_token(M, N, K, A, K, B, bst.COL_MAJOR if b_col_major else bst.ROW_MAJOR,
                             K if b_col_major else N, SA, SB, C, N, ACC, ws, ws_bytes, sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY) and (abuf is None or canary_intact(abuf, CANARY))
    out = decode_out(host(C, np.uint16).reshape(M, N).copy(), "bf16")
    acc = host(ACC, np.int32).reshape(M, N).copy() if with_acc else None
    return out, acc


def oracle_int8_rows(w, rows):
    a = w["a"][rows]
    acc, out = og.gemm_quant_per_token(a, w["b"].T, w["sa"][rows], w["sb"])
    return acc, decode_out(out, "bf16")


@pytest.mark.parametrize("mnk", [(128, 128, 64), (300, 200, 2100), (1, 130, 1024), (257, 129, 40), (520, 700, 3100)])
@pytest.mark.parametrize("bcol", [True, False])
@pytest.mark.parametrize("tile", [(0, 0), (128, 128), (256, 256)])
def test_int8_small(mnk, bcol, tile):
    """Single-CTA 128 x 128 and CTA-pair 256 x 256 tiles (K-chunks of 1024
    folded into exact int32 sums: K = 2100 and 3100 take 3 and 4 chunks)."""
    M, N, K = mnk
    w = wl.int8_per_token(M, N, K, seed=M + K)
    out, acc = run_int8(w, bcol, bst.sched(2, 1, tile_m=tile[0], tile_n=tile[1]))
    racc, rout = oracle_int8_rows(w, np.arange(M))
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)


def test_int8_extreme_sums_exact():
    """All-|127| operands at K=8192 give the largest sums the path must carry
    exactly (8192*127*127 = 132,128,768)."""
    M = N = 128
    K = 8192
    w = wl.int8_per_token(M, N, K, seed=1)
    w["a"][:] = 127
    w["a"][1::2] = -127
    w["b"][:] = 127
    w["b"][:, ::3] = -127
    for tile in [(128, 128), (256, 256)]:
        out, acc = run_int8(w, True, bst.sched(1, 0, tile_m=tile[0], tile_n=tile[1]))
        racc, rout = oracle_int8_rows(w, np.arange(M))
        assert np.array_equal(acc, racc)
        assert_close_fro(out, rout, FRO_MX)


@pytest.mark.parametrize("mnk", [(3001, 1040, 2048), (2432, 1300, 2048)])
def test_int8_bulk_widening_with_and_without_tail(mnk):
    """A is large enough for the bulk-copy widening (at least 2 x SMs x 16 KB
    of int8): 3001 x 2048 leaves a tail of 2048 elements past the last whole
    16 KB chunk for the ordinary-load tail, 2432 x 2048 none.  Every int32
    accumulator bit-exact."""
    M, N, K = mnk
    w = wl.int8_per_token(M, N, K, seed=M + N)
    out, acc = run_int8(w, True)
    racc, rout = oracle_int8_rows(w, np.arange(M))
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)


@functools.lru_cache(maxsize=1)
def _int8_full_oracle():
    w = wl.int8_per_token()
    racc, rout = oracle_int8_rows(w, np.arange(w["M"]))
    return w, racc, rout


def test_int8_full_workload():
    """int8 8192x8192x8192 with per-row / per-column fp32 scales: every int32
    accumulator bit-exact and every dequantised bf16 output within the
    tolerance."""
    w, racc, rout = _int8_full_oracle()
    out, acc = run_int8(w, True)
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)


@pytest.mark.parametrize("S,d", [(1, 0), (8, 1)])
def test_int8_full_workload_without_acc_out(S, d):
    """The call exactly as the bench times it (acc_out = NULL, automatic
    tiles): every bf16 output within the tolerance of the oracle, and
    bit-identical to the same call that also writes the accumulators."""
    w, racc, rout = _int8_full_oracle()
    out, _ = run_int8(w, True, bst.sched(S, d), with_acc=False)
    assert_close_fro(out, rout, FRO_MX)
    out_acc, acc = run_int8(w, True, bst.sched(S, d))
    assert np.array_equal(out.view(np.uint64), out_acc.view(np.uint64))
    assert np.array_equal(acc, racc)


# ------------------------------------------- grouped int8, per-token dequant -

def run_grouped_int8(w, b_col_major=True, sched=None, gdev=None, with_acc=True):
    """One bst_gemm_grouped_quant_per_token call; with_acc=False passes
    acc_out = NULL (the call the bench times) and returns acc None."""
    gm, N, K = w["group_m"], w["N"], w["K"]
    G = len(gm)
    total = sum(gm)
    X = dev(w["x"])
    W = w["w"] if b_col_major else np.ascontiguousarray(np.transpose(w["w"], (0, 2, 1)))   # [G, N, K] or [G, K, N]
    Wd, SA, SB = dev(W), dev(w["sa"]), dev(w["sb"])
    gdev = torch.tensor(gm, dtype=torch.int32, device="cuda") if gdev is None else gdev
    cbuf, C = empty_bytes(max(total, 1) * N * 2, CANARY)
    abuf, ACC = empty_bytes(max(total, 1) * N * 4, CANARY) if with_acc else (None, None)
    ws_bytes = bst.gemm_grouped_quant_per_token_workspace_size(G, total, N, K)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    bst.gemm_grouped_quant_per_token(G, gdev, total, N, K, X, K, Wd, bst.COL_MAJOR if b_col_major else bst.ROW_MAJOR,
                                     K if b_col_major else N, N * K, SA, SB, N, C, N, ACC, ws, ws_bytes, sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY) and (abuf is None or canary_intact(abuf, CANARY))
    out = decode_out(host(C, np.uint16).reshape(-1, N)[:total].copy(), "bf16")
    acc = host(ACC, np.int32).reshape(-1, N)[:total].copy() if with_acc else None
    return out, acc


def oracle_grouped_int8(w, rows=None):
    gm = w["group_m"]
    b = [np.ascontiguousarray(w["w"][g].T) for g in range(len(gm))]     # logical [K, N] per group
    acc, out = og.gemm_grouped_quant_per_token(w["x"], b, gm, w["sa"], w["sb"])
    out = decode_out(out, "bf16")
    return (acc, out) if rows is None else (acc[rows], out[rows])


@pytest.mark.parametrize("gm", [[3, 0, 130, 1, 0, 257], [0, 0, 64], [300], [1] * 9, [300, 0, 513]])
@pytest.mark.parametrize("bcol", [True, False])
def test_grouped_int8_small(gm, bcol):
    """Empty groups, single-row groups, ragged tiles; K = 2100 takes three
    K-chunks of the exact int32 accumulation."""
    w = wl.grouped_int8_per_token(group_m=gm, N=300, K=2100, seed=len(gm) + 7)
    G = len(gm)
    total = sum(gm)
    cap = (-(-total // 256) + G) * -(-300 // 256)
    trace = torch.full((cap * 5,), -1, dtype=torch.int32, device="cuda")
    out, acc = run_grouped_int8(w, bcol, bst.sched(2, 1, trace=trace))
    racc, rout = oracle_grouped_int8(w)
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)
    want = np.array(osw.grouped_swizzle_map(gm, 300, 256, 256, 2, 1), dtype=np.uint32).reshape(-1, 5)
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)[:len(want)]
    assert np.array_equal(tr, want)


def test_grouped_int8_inconsistent_sizes_reported():
    w = wl.grouped_int8_per_token(group_m=[100, 100], N=64, K=64, seed=3)
    gdev = torch.tensor([100, 300], dtype=torch.int32, device="cuda")   # sums past total_m = 200
    with pytest.raises(bst.BstError) as e:
        run_grouped_int8(w, True, gdev=gdev)
    assert e.value.status == bst.ERR_DEVICE
    bst.check_async()      # the error word was cleared


@functools.lru_cache(maxsize=1)
def _grouped_int8_full_oracle(forced):
    w = wl.grouped_int8_per_token(group_m=None if forced is None else list(forced))
    racc, rout = oracle_grouped_int8(w)
    return w, racc, rout


@pytest.mark.parametrize("forced", [None, (0, 2048, 0, 1024, 3072, 0, 2048, 0)])
def test_grouped_int8_full_workload(forced):
    """G = 8 groups summing to 8192 rows, K = N = 4096: every int32
    accumulator bit-exact and every bf16 output within the tolerance; then
    the call as the bench times it (acc_out = NULL), whose outputs must be
    bit-identical to the first call's."""
    w, racc, rout = _grouped_int8_full_oracle(forced)
    out, acc = run_grouped_int8(w, True)
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)
    out_noacc, _ = run_grouped_int8(w, True, bst.sched(1, 0), with_acc=False)
    assert np.array_equal(out_noacc.view(np.uint64), out.view(np.uint64))
