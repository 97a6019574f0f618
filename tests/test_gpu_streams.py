"""Calls on the caller's streams and from several host threads: every launch
goes to the stream passed in, concurrent GEMMs on two streams (split-K CTA
pairs on one, the persistent CTA-pair kernel on the other) both match the
oracle, and host threads issuing their own calls do not disturb each other."""
import threading

import numpy as np
import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from tests.gpu_util import DT, OUT_BYTES, assert_close_f16, decode_out, dev, host
from tests.test_gpu_dense import oracle_dense

pytestmark = pytest.mark.gpu


def _layout(col):
    return bst.COL_MAJOR if col else bst.ROW_MAJOR


def _launch(w, C, stream, sched):
    M, N, K, dt = w["M"], w["N"], w["K"], w["dtype"]
    bst.gemm(M, N, K, w["_A"], DT[dt], _layout(w["a_col_major"]), w["lda"], w["_B"], DT[dt],
             _layout(w["b_col_major"]), w["ldb"], C, DT["f16"], N, sched=sched, stream=stream)


def _result(w, C):
    M, N = w["M"], w["N"]
    raw = host(C, np.uint8).reshape(M, N * OUT_BYTES["f16"]).view(np.uint16)
    return decode_out(raw.copy(), "f16")


def _problem(M, N, K, seed):
    w = wl.dense16(M, N, K, "f16", b_col_major=True, seed=seed, dist="normal")
    w["_A"], w["_B"] = dev(w["a"]), dev(w["b"])
    return w


def test_two_streams_concurrently():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = _problem(1024, 1024, 2048, 21)          # split-K CTA pairs
    w2 = _problem(2048, 1536, 512, 22)           # persistent CTA-pair tiles
    C1 = torch.zeros(w1["M"] * w1["N"], dtype=torch.int16, device="cuda")
    C2 = torch.zeros(w2["M"] * w2["N"], dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        _launch(w1, C1, s1, bst.sched(4, 1))
        _launch(w2, C2, s2, bst.sched(2, 0))
    bst.check_async(s1)
    bst.check_async(s2)
    assert_close_f16(_result(w1, C1), oracle_dense(w1, "f16"))
    assert_close_f16(_result(w2, C2), oracle_dense(w2, "f16"))


def test_launch_goes_to_the_given_stream():
    # the GEMM is ordered after a fill enqueued on the same side stream: if it
    # went to another stream it could read the operand before the fill
    s = torch.cuda.Stream()
    w = _problem(300, 260, 320, 23)
    A2 = torch.empty_like(w["_A"])
    C = torch.zeros(w["M"] * w["N"], dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)              # keep the side stream busy before the copy
        A2.copy_(w["_A"])
    w["_A"] = A2
    _launch(w, C, s, bst.sched(1, 0))
    bst.check_async(s)
    assert_close_f16(_result(w, C), oracle_dense(w, "f16"))


def test_host_threads_issue_their_own_calls():
    probs = [_problem(256 + 64 * i, 384, 256 + 128 * i, 30 + i) for i in range(4)]
    outs = [torch.zeros(p["M"] * p["N"], dtype=torch.int16, device="cuda") for p in probs]
    # the same calls from this thread first
    for i, (p, C) in enumerate(zip(probs, outs)):
        _launch(p, C, torch.cuda.current_stream(), bst.sched(1 + i, i % 2))
    bst.check_async()
    for p, C in zip(probs, outs):
        assert_close_f16(_result(p, C), oracle_dense(p, "f16"))
        C.zero_()
    torch.cuda.synchronize()
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    _launch(probs[i], outs[i], s, bst.sched(1 + i, i % 2))
            s.synchronize()
        except Exception as e:        # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    bst.check_async()
    for p, C in zip(probs, outs):
        assert_close_f16(_result(p, C), oracle_dense(p, "f16"))
