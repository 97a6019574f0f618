"""GPU parity of the fp16/bf16 path (bst_gemm, bst_gemm_batched) and of the
device scheduler (bst_swizzle_map) against the CPU oracle."""
import functools
import itertools

import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from oracle import gemm as og, swizzle as osw
from tests.gpu_util import (DT, FRO_F16, OUT_BYTES, assert_close_f16, assert_special_equal, canary_intact,
                            decode_out, dev, empty_bytes, host)
from tests.swizzle_checks import check_map

pytestmark = pytest.mark.gpu
CANARY = 256


def _layout(col):
    return bst.COL_MAJOR if col else bst.ROW_MAJOR


def run_dense(w, out="f16", sched=None, ldc=None):
    M, N, K, dt = w["M"], w["N"], w["K"], w["dtype"]
    ldc = N if ldc is None else ldc
    A = dev(w["a"])
    B = dev(w["b"])
    cbuf, C = empty_bytes(max(M * ldc, 1) * OUT_BYTES[out], CANARY)
    bst.gemm(M, N, K, A, DT[dt], _layout(w["a_col_major"]), w["lda"], B, DT[dt], _layout(w["b_col_major"]),
             w["ldb"], C, DT[out], ldc, sched=sched)
    bst.check_async()
    assert canary_intact(cbuf, CANARY), "write outside C"
    rows = host(C, np.uint8).reshape(M, ldc * OUT_BYTES[out])
    assert (rows[:, N * OUT_BYTES[out]:] == 0x5A).all(), "write into the padding between N and ldc"
    raw = rows.view(np.float32 if out == "f32" else np.uint16)[:, :N]
    return decode_out(raw.copy(), out)


def oracle_dense(w, out="f16"):
    M, N, K, dt = w["M"], w["N"], w["K"], w["dtype"]
    a = og.as_logical(og.decode(w["a"], dt), M, K, w["lda"], w["a_col_major"])
    b = og.as_logical(og.decode(w["b"], dt), K, N, w["ldb"], w["b_col_major"])
    return decode_out(og.gemm(a, b, out), out)


# ------------------------------------------------------------ scheduler ---

MAP_SHAPES = [(500, 380, 128, 128, 1), (1024, 1024, 128, 64, 1), (8192, 8192, 128, 256, 1),
              (129, 2000, 128, 64, 3), (48, 74, 16, 16, 2), (1, 1, 128, 128, 1), (1000, 37, 16, 8, 1)]


@pytest.mark.parametrize("shape", MAP_SHAPES)
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8, 9, 100000])
@pytest.mark.parametrize("d", [0, 1])
def test_swizzle_map_bit_exact(shape, S, d):
    M, N, tm, tn, batch = shape
    want = np.array(osw.swizzle_map(M, N, tm, tn, S, d, batch=batch), dtype=np.uint32)
    out = torch.zeros(want.size, dtype=torch.int32, device="cuda")
    bst.swizzle_map(M, N, tm, tn, batch, bst.sched(S, d), out)
    bst.check_async()
    got = out.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(got, want)
    core = len(want) // batch
    assert check_map([tuple(r[1:]) for r in got[:core]], M, N, tm, tn, S, d) == []


@pytest.mark.parametrize("gm", [[0, 300, 0, 129, 1, 0, 1024], [8192], [0, 0, 5], [1] * 40])
@pytest.mark.parametrize("S,d", [(1, 0), (2, 0), (3, 1), (8, 1)])
def test_swizzle_map_grouped_bit_exact(gm, S, d):
    N, tm, tn = 700, 128, 128
    want = np.array(osw.grouped_swizzle_map(gm, N, tm, tn, S, d), dtype=np.uint32).reshape(-1, 5)
    gdev = torch.tensor(gm, dtype=torch.int32, device="cuda")
    cap = max(len(want), 1)
    out = torch.full((cap * 5,), -1, dtype=torch.int32, device="cuda")
    bst.swizzle_map_grouped(len(gm), gdev, N, tm, tn, bst.sched(S, d), out, cap)
    bst.check_async()
    got = out.cpu().numpy().view(np.uint32).reshape(-1, 5)[:len(want)]
    assert np.array_equal(got, want)


# ---------------------------------------------------------- fp16 tail ------

@pytest.mark.parametrize("d", [0, 1])
def test_fp16_tail_workload(d):
    """fp16 500x380x256 row-major A and B, 128x128 tiles, SwizzleOffset 3."""
    w = wl.fp16_tail()
    ntiles = 4 * 3
    trace = torch.zeros(ntiles * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, "f16", bst.sched(3, d, tile_n=128, tile_m=128, trace=trace))
    assert_close_f16(got, oracle_dense(w, "f16"))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(500, 380, 128, 128, 3, d), dtype=np.uint32))


# -------------------------------------------------------- fp16 square ------

@pytest.mark.parametrize("S", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [0, 1])
def test_fp16_square_workload(S, d):
    """fp16 1024x1024x2048, A row-major, B column-major, N(0,1)/sqrt(K)."""
    w = wl.fp16_square()
    got = run_dense(w, "f16", bst.sched(S, d))
    assert_close_f16(got, oracle_dense(w, "f16"))


def test_fp16_square_trace_per_tile_width():
    w = wl.fp16_square()
    ref = oracle_dense(w, "f16")
    for tn in (64, 128, 256):
        tiles = 8 * (1024 // tn)
        trace = torch.zeros(tiles * 5, dtype=torch.int32, device="cuda")
        got = run_dense(w, "f16", bst.sched(2, 0, tile_n=tn, tile_m=128, trace=trace))
        assert_close_f16(got, ref)
        tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
        assert np.array_equal(tr, np.array(osw.swizzle_map(1024, 1024, 128, tn, 2, 0), dtype=np.uint32))


# ------------------------------------------------- shapes and layouts ------

SMALL = [(1, 1, 16), (127, 129, 72), (128, 128, 64), (129, 127, 200), (500, 64, 256), (64, 500, 24),
         (257, 300, 1000)]


@pytest.mark.parametrize("mnk", SMALL)
@pytest.mark.parametrize("acol,bcol", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_small_shapes_layouts(mnk, acol, bcol, dt):
    M, N, K = mnk
    w = wl.dense16(M, N, K, dt, a_col_major=acol, b_col_major=bcol, seed=M * 7 + N + K)
    for tn in (64, 128, 256):
        got = run_dense(w, dt, bst.sched(2, 0, tile_n=tn))
        assert_close_f16(got, oracle_dense(w, dt))


@pytest.mark.parametrize("out", ["f16", "bf16", "f32"])
def test_output_types(out):
    w = wl.dense16(300, 260, 320, "bf16", seed=3)
    got = run_dense(w, out, bst.sched(1, 1))
    assert_close_f16(got, oracle_dense(w, out))


@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad", [(3, 0, 0), (0, 5, 0), (1, 1, 3), (8, 8, 8)])
def test_padded_and_unaligned_leading_dims(lda_pad, ldb_pad, ldc_pad):
    """Odd leading dimensions take the ordinary-load path (TMA needs 16-byte
    pitches); both paths must give the same result."""
    M, N, K = 200, 190, 136
    w = wl.dense16(M, N, K, "f16", b_col_major=False, seed=5, lda=K + lda_pad, ldb=N + ldb_pad)
    got = run_dense(w, "f16", bst.sched(3, 0), ldc=N + ldc_pad)
    assert_close_f16(got, oracle_dense(w, "f16"))


@pytest.mark.parametrize("tn", [64, 128, 256])
@pytest.mark.parametrize("acol,lda_pad,ldb_pad", [(False, 0, 4), (False, 0, 1), (True, 4, 0), (False, 3, 3)])
def test_copied_operands_several_tiles_per_cta(tn, acol, lda_pad, ldb_pad):
    """Operands TMA cannot fetch (8-byte and 2-byte aligned pitches), with
    fewer CTAs than tiles and more k-blocks than ring stages: the epilogue
    warps help copy only each CTA's first tile, and on the later tiles the
    load warps arrive for them."""
    M, N, K = 700, 520, 1100
    w = wl.dense16(M, N, K, "f16", a_col_major=acol, b_col_major=False, seed=tn + lda_pad * 5 + ldb_pad,
                   lda=(M if acol else K) + lda_pad, ldb=N + ldb_pad)
    got = run_dense(w, "f16", bst.sched(2, 1, tile_n=tn, num_ctas=5))
    assert_close_f16(got, oracle_dense(w, "f16"))


ROWS2 = [(500, 380, 256, 0), (300, 300, 1000, 0), (129, 60, 64, 0), (257, 500, 130, 0), (64, 132, 2, 0),
         (500, 380, 256, 8), (200, 76, 255, 0), (70, 4, 66, 0), (33, 12, 130, 0)]


@pytest.mark.parametrize("mnk_pad", ROWS2)
@pytest.mark.parametrize("dt,out", [("f16", "f16"), ("bf16", "f32")])
@pytest.mark.parametrize("kw", [{}, {"num_ctas": 3}, {"shuffle_k": 1}])
def test_b_through_two_row_view(mnk_pad, dt, out, kw):
    """Row-major B whose pitch is 8 bytes off a multiple of 16 (ldb = 4 mod 8)
    goes through the two-row tensor-map view with 128 x 64 tiles: ragged N and
    K tails, K = 2, several tiles per CTA, ShuffleK; an odd K (255) takes the
    copy path instead."""
    M, N, K, pad = mnk_pad
    w = wl.dense16(M, N, K, dt, b_col_major=False, seed=M + N + K + pad, ldb=N + pad, dist="normal")
    assert w["ldb"] % 8 == 4
    lm, ln = -(-M // 128), -(-N // 64)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, out, bst.sched(2, 1, trace=trace, **kw))
    assert_close_f16(got, oracle_dense(w, out))
    if K % 2 == 0:
        tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
        assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 128, 64, 2, 1), dtype=np.uint32))


@pytest.mark.parametrize("mnk", [(256, 380, 128), (136, 124, 320)])
def test_b_two_row_view_with_column_major_a(mnk):
    """The two-row view of B beside an MN-major (column-major) A loaded by TMA
    in 64-row atoms, with an output pitch that is not 16-byte aligned."""
    M, N, K = mnk
    w = wl.dense16(M, N, K, "f16", a_col_major=True, b_col_major=False, seed=M + K, dist="normal")
    assert w["ldb"] % 8 == 4 and (w["lda"] * 2) % 16 == 0
    got = run_dense(w, "f16", bst.sched(1, 0), ldc=N + 3)
    assert_close_f16(got, oracle_dense(w, "f16"))


@pytest.mark.parametrize("tm", [128, 256])
@pytest.mark.parametrize("out,ldc_pad", [("f16", 1), ("f16", 2), ("bf16", 4), ("f16", 8), ("f32", 1), ("f32", 2),
                                         ("f32", 4)])
def test_output_pitch_vector_widths(tm, out, ldc_pad):
    """Every output pitch (2-, 4-, 8- and 16-byte aligned rows) goes through the
    staged epilogue's widest legal store; the padding columns stay untouched."""
    M, N, K = 333, 290, 200
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=ldc_pad + tm, lda=208, ldb=208)
    got = run_dense(w, out, bst.sched(2, 1, tile_m=tm), ldc=N + ldc_pad)
    assert_close_f16(got, oracle_dense(w, out))


def test_k_zero_writes_zeros_and_empty_is_noop():
    w = wl.dense16(70, 50, 0, "f16", seed=1, lda=1)
    got = run_dense(w, "f32")
    assert not got.any()
    cbuf, C = empty_bytes(64, CANARY)
    bst.gemm(0, 10, 10, None, bst.F16, bst.ROW_MAJOR, 10, None, bst.F16, bst.ROW_MAJOR, 10, C, bst.F16, 10)
    bst.gemm(10, 0, 10, None, bst.F16, bst.ROW_MAJOR, 10, None, bst.F16, bst.ROW_MAJOR, 10, C, bst.F16, 10)
    bst.check_async()
    assert (C == 0x5A).all().item()


def test_special_values_identity_and_zero():
    M = 256
    eye = np.eye(M, dtype=np.float16).view(np.uint16)
    w = wl.dense16(M, M, M, "f16", seed=2)
    w_id = dict(w, b=eye, ldb=M, b_col_major=False)
    got = run_dense(w_id, "f16")
    assert np.array_equal(got, decode_out(w["a"].copy(), "f16"))   # A.I == A exactly
    w_zero = dict(w, b=np.zeros_like(eye))
    assert not run_dense(w_zero, "f32").any()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_special_values_inf_nan_and_overflow(dt):
    """IEEE special values through the fp32 accumulation and the output cast:
    an infinity in row 3 of A makes that row +-inf, with NaN where it meets a
    zero of B (inf x 0); a NaN makes row 7 NaN; for fp16, a row of 65504s
    makes sums past the fp16 range round to +-inf.  NaN and infinity positions
    (with signs) equal the oracle's; the finite rest is within the tolerance."""
    M, N, K = 256, 256, 128
    w = wl.dense16(M, N, K, dt, seed=9)
    inf, nan, big = (0x7C00, 0x7E00, 0x7BFF) if dt == "f16" else (0x7F80, 0x7FC0, None)
    a, b = w["a"].copy(), w["b"].copy()          # row-major [M, K] and [K, N] bit patterns
    a[3, 10] = inf
    a[7, 20] = nan
    b[10, 9] = 0
    if big is not None:
        a[11, :] = big
        b[:, 5] = big
    got = run_dense(dict(w, a=a, b=b), dt)
    # the plain definition summed without BLAS (whose kernels need not keep
    # IEEE infinities and NaNs), rounded once by the oracle
    acc = np.einsum("ik,kj->ij", og.decode(a, dt), og.decode(b, dt))
    ref = decode_out(og.round_out(acc, dt), dt)
    assert np.isnan(ref[7]).all() and np.isnan(ref[3, 9]) and np.isinf(ref[3, 0])
    assert_special_equal(got, ref, FRO_F16)


# ------------------------------------------------------------- batched -----

@pytest.mark.parametrize("acol,bcol", [(False, True), (True, False)])
def test_batched(acol, bcol):
    M, N, K, batch = 200, 136, 264, 3
    w = wl.dense16(M, N, K, "bf16", a_col_major=acol, b_col_major=bcol, seed=9, batch=batch)
    A = dev(w["a"])
    B = dev(w["b"])
    sa = w["a"][0].size
    sb = w["b"][0].size
    cbuf, C = empty_bytes(batch * M * N * 2, CANARY)
    trace_tiles = batch * 2 * 2
    trace = torch.zeros(trace_tiles * 5, dtype=torch.int32, device="cuda")
    bst.gemm_batched(M, N, K, A, bst.BF16, _layout(acol), w["lda"], sa, B, bst.BF16, _layout(bcol), w["ldb"], sb,
                     C, bst.BF16, N, M * N, batch, sched=bst.sched(1, 0, tile_n=128, tile_m=128, trace=trace))
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    got = decode_out(host(C, np.uint16).reshape(batch, M, N).copy(), "bf16")
    for i in range(batch):
        a = og.as_logical(og.decode(w["a"][i], "bf16"), M, K, w["lda"], acol)
        b = og.as_logical(og.decode(w["b"][i], "bf16"), K, N, w["ldb"], bcol)
        assert_close_f16(got[i], decode_out(og.gemm(a, b, "bf16"), "bf16"))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 128, 128, 1, 0, batch=batch), dtype=np.uint32))


@pytest.mark.parametrize("tm", [128, 256])
def test_batched_unaligned_c_batch_stride(tm):
    """A C batch stride of an odd number of elements limits every store to
    2 bytes; the gaps between the batches stay untouched."""
    M, N, K, batch = 150, 100, 128, 3
    gap = 3
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=10, batch=batch)
    A, B = dev(w["a"]), dev(w["b"])
    sc = M * N + gap
    cbuf, C = empty_bytes(batch * sc * 2, CANARY)
    bst.gemm_batched(M, N, K, A, bst.F16, bst.ROW_MAJOR, w["lda"], w["a"][0].size, B, bst.F16, bst.COL_MAJOR,
                     w["ldb"], w["b"][0].size, C, bst.F16, N, sc, batch, sched=bst.sched(2, 0, tile_m=tm))
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    raw = host(C, np.uint8)
    for i in range(batch):
        blk = raw[i * sc * 2:(i * sc + M * N) * 2]
        assert (raw[(i * sc + M * N) * 2:(i + 1) * sc * 2] == 0x5A).all()
        got = decode_out(blk.view(np.uint16).reshape(M, N).copy(), "f16")
        a = og.as_logical(og.decode(w["a"][i], "f16"), M, K, w["lda"], False)
        b = og.as_logical(og.decode(w["b"][i], "f16"), K, N, w["ldb"], True)
        assert_close_f16(got, decode_out(og.gemm(a, b, "f16"), "f16"))


# ------------------------------------------------- CTA-pair (256-row) ------

PAIR_SHAPES = [(256, 256, 64), (300, 200, 136), (513, 384, 1000), (1, 136, 72)]


@pytest.mark.parametrize("mnk", PAIR_SHAPES)
@pytest.mark.parametrize("acol,bcol", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("tn", [128, 256])
def test_pair_shapes_layouts(mnk, acol, bcol, tn):
    M, N, K = mnk
    up8 = lambda x: -(-x // 8) * 8           # 16-byte pitches, so both operands can use TMA
    w = wl.dense16(M, N, K, "bf16", a_col_major=acol, b_col_major=bcol, seed=M + 3 * N + K,
                   lda=up8(M if acol else K), ldb=up8(K if bcol else N))
    lm, ln = -(-M // 256), -(-N // tn)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, "bf16", bst.sched(2, 1, tile_n=tn, tile_m=256, trace=trace))
    assert_close_f16(got, oracle_dense(w, "bf16"))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 256, tn, 2, 1), dtype=np.uint32))


@pytest.mark.parametrize("S,d", [(1, 0), (2, 0), (4, 1), (8, 1)])
def test_pair_fp16_square_workload(S, d):
    w = wl.fp16_square()
    trace = torch.zeros(16 * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, "f16", bst.sched(S, d, tile_n=256, tile_m=256, trace=trace))
    assert_close_f16(got, oracle_dense(w, "f16"))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(1024, 1024, 256, 256, S, d), dtype=np.uint32))


@functools.lru_cache(maxsize=1)
def _large_bf16():
    w = wl.dense16(8192, 2048, 8192, "bf16", b_col_major=True, seed=81)
    return w, oracle_dense(w, "bf16")


@pytest.mark.parametrize("S,d", [(1, 1), (8, 1), (4, 0)])
def test_pair_large_operands_several_waves(S, d):
    """bf16 8192 x 2048 x 8192 on CTA-pair tiles: 256 tiles over the 76 pairs of
    the persistent grid (several waves), operands of 134 and 33.5 MB, both
    window directions.  Every element within the tolerance of the oracle."""
    w, ref = _large_bf16()
    assert_close_f16(run_dense(w, "bf16", bst.sched(S, d)), ref)


def test_pair_needs_tma_operands():
    """A CTA pair fetches both operands with TMA; forcing it on a 260-byte
    pitch is refused instead of silently changing the schedule."""
    w = wl.dense16(64, 130, 72, "f16", b_col_major=False, seed=1)
    with pytest.raises(bst.BstError) as e:
        run_dense(w, "f16", bst.sched(1, 0, tile_m=256))
    assert e.value.status == bst.ERR_UNSUPPORTED
    assert_close_f16(run_dense(w, "f16", bst.sched(1, 0)), oracle_dense(w, "f16"))


def test_pair_batched():
    M, N, K, batch = 300, 256, 200, 3
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=4, batch=batch)
    A, B = dev(w["a"]), dev(w["b"])
    cbuf, C = empty_bytes(batch * M * N * 2, CANARY)
    bst.gemm_batched(M, N, K, A, bst.F16, bst.ROW_MAJOR, w["lda"], w["a"][0].size, B, bst.F16, bst.COL_MAJOR,
                     w["ldb"], w["b"][0].size, C, bst.F16, N, M * N, batch, sched=bst.sched(1, 0, tile_m=256))
    bst.check_async()
    assert canary_intact(cbuf, CANARY)
    got = decode_out(host(C, np.uint16).reshape(batch, M, N).copy(), "f16")
    for i in range(batch):
        a = og.as_logical(og.decode(w["a"][i], "f16"), M, K, w["lda"], False)
        b = og.as_logical(og.decode(w["b"][i], "f16"), K, N, w["ldb"], True)
        assert_close_f16(got[i], decode_out(og.gemm(a, b, "f16"), "f16"))


# ------------------------------------------------- split-K CTA pairs -------

@pytest.mark.parametrize("mnk", [(256, 256, 512), (300, 500, 1000), (1024, 1024, 2048), (17, 260, 4096)])
@pytest.mark.parametrize("acol,bcol", [(False, True), (True, False), (False, False), (True, True)])
@pytest.mark.parametrize("splits", [2, 4])
@pytest.mark.parametrize("tn", [256, 128])
def test_splitk_shapes_layouts(mnk, acol, bcol, splits, tn):
    M, N, K = mnk
    up8 = lambda x: -(-x // 8) * 8
    w = wl.dense16(M, N, K, "f16", a_col_major=acol, b_col_major=bcol, seed=M + N + K + splits,
                   lda=up8(M if acol else K), ldb=up8(K if bcol else N), dist="normal")
    lm, ln = -(-M // 256), -(-N // tn)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, "f16", bst.sched(3, 1, split_k=splits, tile_n=tn, trace=trace))
    assert_close_f16(got, oracle_dense(w, "f16"))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 256, tn, 3, 1), dtype=np.uint32))


@pytest.mark.parametrize("tn,splits", [(256, 2), (128, 2), (128, 4)])
@pytest.mark.parametrize("out,ldc_pad", [("f16", 1), ("bf16", 2), ("f16", 4), ("f32", 1), ("f32", 2)])
def test_splitk_output_pitches(tn, splits, out, ldc_pad):
    M, N, K = 300, 270, 1024
    w = wl.dense16(M, N, K, "bf16", b_col_major=True, seed=tn + splits, dist="normal")
    got = run_dense(w, out, bst.sched(2, 0, split_k=splits, tile_n=tn), ldc=N + ldc_pad)
    assert_close_f16(got, oracle_dense(w, out))


def test_splitk_auto_choice_matches_oracle():
    # the headline shape with the automatic split choice (and the timeline debug output)
    w = wl.fp16_square()
    tl = torch.zeros(160 * 64, dtype=torch.int64, device="cuda")
    got = run_dense(w, "f16", bst.sched(1, 1, timeline=tl))
    assert_close_f16(got, oracle_dense(w, "f16"))


@pytest.mark.parametrize("tn,splits", [(64, 2), (128, 2), (128, 4)])
@pytest.mark.parametrize("mnk,acol,lda_pad,ldb_pad", [((500, 380, 256), False, 0, 0), ((300, 200, 1000), True, 4, 3),
                                                      ((129, 127, 200), False, 3, 0), ((64, 90, 64), False, 0, 0)])
@pytest.mark.parametrize("out", ["f16", "f32"])
def test_copied_operands_split_k(tn, splits, mnk, acol, lda_pad, ldb_pad, out):
    """One-CTA split-K for operands TMA cannot fetch (8- and 2-byte aligned
    pitches): the partials of a cluster's CTAs summed by column ownership,
    the tile order still the scheduler's; K = 64 leaves splits without
    k-blocks."""
    M, N, K = mnk
    w = wl.dense16(M, N, K, "bf16", a_col_major=acol, b_col_major=False, seed=M + N + K + tn + splits,
                   lda=(M if acol else K) + lda_pad, ldb=N + ldb_pad, dist="normal")
    lm, ln = -(-M // 128), -(-N // tn)
    trace = torch.zeros(lm * ln * 5, dtype=torch.int32, device="cuda")
    got = run_dense(w, out, bst.sched(3, 1, split_k=splits, tile_n=tn, tile_m=128, trace=trace))
    assert_close_f16(got, oracle_dense(w, out))
    tr = trace.cpu().numpy().view(np.uint32).reshape(-1, 5)
    assert np.array_equal(tr, np.array(osw.swizzle_map(M, N, 128, tn, 3, 1), dtype=np.uint32))


def test_splitk_more_splits_than_kblocks_and_f32_out():
    # K = 64: one k-block, four splits -> three splits contribute zeros
    w = wl.dense16(256, 256, 64, "bf16", b_col_major=True, seed=8)
    got = run_dense(w, "f32", bst.sched(1, 0, split_k=4))
    assert_close_f16(got, oracle_dense(w, "f32"))
