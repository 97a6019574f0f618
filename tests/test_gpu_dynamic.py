"""GPU parity of the two scheduling options of bst_sched against the CPU
oracle: dynamic task allocation (clusters claiming not-yet-started clusters'
tasks through cluster launch control) and ShuffleK (a per-task rotated K
start).  Every path that takes them (plain, batched, grouped slice-M,
slice-K, int8) must give the oracle's results, and the per-task trace must
still be the scheduler's map: each task computed, with its own tile."""
import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from oracle import gemm as og, swizzle as osw
from tests.gpu_util import FRO_MX, assert_close_f16, assert_close_fro, decode_out
from tests.test_gpu_dense import oracle_dense, run_dense
from tests.test_gpu_slice_k import check_groups, make, oracle_slice_k, run_slice_k
from tests.test_gpu_variants import oracle_int8_rows, run_grouped, run_grouped_int8, run_int8, run_mx

pytestmark = pytest.mark.gpu


def _trace(tasks):
    return torch.full((tasks * 5,), -1, dtype=torch.int32, device="cuda")


def _rows(trace):
    return trace.cpu().numpy().view(np.uint32).reshape(-1, 5)


@pytest.mark.parametrize("mnk", [(1024, 1024, 2048), (520, 700, 3096), (257, 300, 1000), (1, 1, 16), (2048, 384, 64)])
@pytest.mark.parametrize("tn", [128, 256])
@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (0, 1), (1, 1)])
def test_dense_pair(mnk, tn, dyn, shuffle):
    M, N, K = mnk
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=M + N + K)
    tiles = -(-M // 256) * -(-N // tn)
    trace = _trace(tiles)
    got = run_dense(w, "f16", bst.sched(2, 1, tile_n=tn, tile_m=256, trace=trace, dynamic=dyn, shuffle_k=shuffle))
    assert_close_f16(got, oracle_dense(w, "f16"))
    assert np.array_equal(_rows(trace), np.array(osw.swizzle_map(M, N, 256, tn, 2, 1), dtype=np.uint32))


@pytest.mark.parametrize("tn,splits", [(256, 2), (128, 2), (256, 4), (128, 4)])
@pytest.mark.parametrize("mnk", [(1024, 1024, 2048), (300, 500, 1000), (256, 256, 200)])
def test_shuffle_k_split_k(tn, splits, mnk):
    """Split-K tiles rotate within each split's K range (K = 200 leaves
    splits of 0 or 1 k-blocks)."""
    M, N, K = mnk
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=M + K + tn)
    got = run_dense(w, "f16", bst.sched(1, 0, tile_n=tn, tile_m=256, split_k=splits, shuffle_k=1))
    assert_close_f16(got, oracle_dense(w, "f16"))


@pytest.mark.parametrize("mnk,lda_pad", [((300, 260, 1000), 0), ((129, 500, 300), 3), ((640, 128, 4096), 0)])
@pytest.mark.parametrize("tn", [64, 128, 256])
def test_shuffle_k_one_cta(mnk, lda_pad, tn):
    """One-CTA tiles, through TMA and (lda not 16-byte aligned) through the
    register-staged loader."""
    M, N, K = mnk
    w = wl.dense16(M, N, K, "bf16", seed=M + K, lda=K + lda_pad)
    got = run_dense(w, "bf16", bst.sched(1, 0, tile_n=tn, tile_m=128, shuffle_k=1))
    assert_close_f16(got, oracle_dense(w, "bf16"))


def test_dynamic_auto_tile_and_many_calls():
    """Dynamic with the automatic tile width, 20 calls back to back on one
    stream (no state carries from one launch to the next)."""
    w = wl.fp16_square()
    ref = oracle_dense(w, "f16")
    for _ in range(3):
        got = run_dense(w, "f16", bst.sched(8, 1, dynamic=1))
    assert_close_f16(got, ref)
    A = torch.from_numpy(np.ascontiguousarray(w["a"]).view(np.uint8).reshape(-1).copy()).cuda()
    B = torch.from_numpy(np.ascontiguousarray(w["b"]).view(np.uint8).reshape(-1).copy()).cuda()
    C = torch.zeros(1024 * 1024, dtype=torch.int16, device="cuda")
    for i in range(20):
        bst.gemm(1024, 1024, 2048, A, bst.F16, bst.ROW_MAJOR, 2048, B, bst.F16, bst.COL_MAJOR, 2048, C, bst.F16,
                 1024, sched=bst.sched(1 + i % 4, i % 2, dynamic=1, shuffle_k=i % 2))
    bst.check_async()
    assert_close_f16(decode_out(C.cpu().numpy().view(np.uint16).reshape(1024, 1024), "f16"), ref)


@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (0, 1), (1, 1)])
def test_batched(dyn, shuffle):
    M, N, K, batch = 300, 264, 520, 3
    w = wl.dense16(M, N, K, "bf16", b_col_major=True, seed=11, batch=batch)
    A = torch.from_numpy(np.ascontiguousarray(w["a"]).view(np.uint8).reshape(-1).copy()).cuda()
    B = torch.from_numpy(np.ascontiguousarray(w["b"]).view(np.uint8).reshape(-1).copy()).cuda()
    C = torch.zeros(batch * M * N, dtype=torch.int16, device="cuda")
    tiles = batch * 2 * 2
    trace = _trace(tiles)
    bst.gemm_batched(M, N, K, A, bst.BF16, bst.ROW_MAJOR, w["lda"], w["a"][0].size, B, bst.BF16, bst.COL_MAJOR,
                     w["ldb"], w["b"][0].size, C, bst.BF16, N, M * N, batch,
                     sched=bst.sched(1, 0, tile_n=256, tile_m=256, trace=trace, dynamic=dyn, shuffle_k=shuffle))
    bst.check_async()
    got = decode_out(C.cpu().numpy().view(np.uint16).reshape(batch, M, N), "bf16")
    for i in range(batch):
        a = og.as_logical(og.decode(w["a"][i], "bf16"), M, K, w["lda"], False)
        b = og.as_logical(og.decode(w["b"][i], "bf16"), K, N, w["ldb"], True)
        assert_close_f16(got[i], decode_out(og.gemm(a, b, "bf16"), "bf16"))
    assert np.array_equal(_rows(trace), np.array(osw.swizzle_map(M, N, 256, 256, 1, 0, batch=batch), dtype=np.uint32))


@pytest.mark.parametrize("gm", [[3, 0, 130, 1, 0, 600], [0, 0, 64], [1] * 9])
@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (0, 1), (1, 1)])
def test_grouped_slice_m(gm, dyn, shuffle):
    """The grid of a dynamic grouped launch is a bound on the task count
    (the tasks are counted on the device): clusters past the end find no
    task."""
    w = wl.grouped_bf16(group_m=gm, N=296, K=264, seed=len(gm))
    total = sum(gm)
    cap = (-(-total // 256) + len(gm)) * -(-296 // 256)
    trace = _trace(cap)
    got = run_grouped(w, bst.sched(2, 0, tile_n=256, tile_m=256, trace=trace, dynamic=dyn, shuffle_k=shuffle))
    ref = decode_out(og.gemm_grouped(og.decode(w["x"], "bf16"), og.decode(w["w"], "bf16"), gm, "bf16"), "bf16")
    assert_close_f16(got, ref)
    want = np.array(osw.grouped_swizzle_map(gm, 296, 256, 256, 2, 0), dtype=np.uint32).reshape(-1, 5)
    assert np.array_equal(_rows(trace)[:len(want)], want)


@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (0, 1), (1, 1)])
def test_slice_k(dyn, shuffle):
    gk = [1, 0, 63, 300, 0, 129]
    M, N = 600, 520
    a, b = make(gk, M, N, seed=21)
    tiles = len(gk) * 3 * 3
    trace = _trace(tiles)
    got = run_slice_k(a, b, gk, False, True, sched=bst.sched(3, 1, tile_n=256, trace=trace, dynamic=dyn,
                                                                shuffle_k=shuffle))
    check_groups(got, oracle_slice_k(a, b, gk, "bf16", "bf16"), gk)
    assert np.array_equal(_rows(trace), np.array(osw.swizzle_map(M, N, 256, 256, 3, 1, batch=len(gk)),
                                                 dtype=np.uint32))


@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (0, 1), (1, 1)])
def test_int8(dyn, shuffle):
    """Exact int32 accumulators: K = 3100 takes four exact K-chunks, and with
    ShuffleK the chunks hold rotated k-blocks."""
    w = wl.int8_per_token(M=520, N=700, K=3100, seed=5)
    out, acc = run_int8(w, True, bst.sched(1, 0, tile_m=256, tile_n=256, dynamic=dyn, shuffle_k=shuffle))
    racc, rout = oracle_int8_rows(w, np.arange(520))
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)


def test_int8_shuffle_one_cta():
    w = wl.int8_per_token(M=300, N=200, K=2100, seed=6)
    out, acc = run_int8(w, False, bst.sched(1, 0, tile_m=128, tile_n=128, shuffle_k=1))
    racc, rout = oracle_int8_rows(w, np.arange(300))
    assert np.array_equal(acc, racc)
    assert_close_fro(out, rout, FRO_MX)


@pytest.mark.parametrize("dyn,shuffle", [(1, 0), (1, 1)])
def test_grouped_int8(dyn, shuffle):
    gm = [3, 0, 300, 1, 0, 513]
    w = wl.grouped_int8_per_token(group_m=gm, N=300, K=2100, seed=9)
    out, acc = run_grouped_int8(w, True, bst.sched(2, 1, dynamic=dyn, shuffle_k=shuffle))
    b = [np.ascontiguousarray(w["w"][g].T) for g in range(len(gm))]
    racc, rout = og.gemm_grouped_quant_per_token(w["x"], b, gm, w["sa"], w["sb"])
    assert np.array_equal(acc, racc)
    assert_close_fro(out, decode_out(rout, "bf16"), FRO_MX)


def test_flags_rejected():
    """MXFP8 takes neither option; dynamic needs CTA-pair tiles and its own
    grid; neither combines with split-K.  Nothing is launched."""
    w = wl.mxfp8(128, 128, 256, seed=1)
    for kw in ({"dynamic": 1}, {"shuffle_k": 1}):
        with pytest.raises(bst.BstError) as e:
            run_mx(w, bst.sched(1, 0, **kw))
        assert e.value.status == bst.ERR_UNSUPPORTED
    d = wl.dense16(256, 256, 256, "f16", b_col_major=True, seed=2)
    for kw, status in (({"dynamic": 1, "num_ctas": 8}, bst.ERR_INVALID_ARG),
                       ({"dynamic": 1, "tile_m": 128}, bst.ERR_UNSUPPORTED),
                       ({"dynamic": 1, "split_k": 2}, bst.ERR_UNSUPPORTED),
                       ({"dynamic": 2}, bst.ERR_INVALID_ARG)):
        with pytest.raises(bst.BstError) as e:
            run_dense(d, "f16", bst.sched(1, 0, **kw))
        assert e.value.status == status
    bst.check_async()
