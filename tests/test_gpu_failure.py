"""Device-side failure detection without a GPU fault: a bounded wait that
nothing completes gives up after its limit, the error word reports
BST_ERR_TIMEOUT through bst_check_async, and the device stays usable.

The wait runs in bst_wait_check's one-CTA kernel, on a shared-memory barrier
with nothing asynchronous in flight, through the same bounded wait the GEMM
kernels use between their roles."""
import time

import pytest
import torch

import block_swizzled_tile_gb300 as bst
from block_swizzled_tile_gb300 import workloads as wl
from tests.test_gpu_dense import oracle_dense, run_dense
from tests.gpu_util import assert_close_f16

pytestmark = pytest.mark.gpu


def test_wait_that_completes_reports_ok():
    bst.wait_check(1_000_000, arrive=True)
    bst.check_async()


def test_wait_that_nothing_completes_times_out():
    t0 = time.perf_counter()
    bst.wait_check(2_000_000, arrive=False)          # 2 ms limit
    with pytest.raises(bst.BstError) as e:
        bst.check_async()
    assert e.value.status == bst.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the error word was read and cleared: the next check is clean
    bst.check_async()


def test_device_usable_after_a_timeout():
    bst.wait_check(1_000_000, arrive=False)
    with pytest.raises(bst.BstError) as e:
        bst.check_async()
    assert e.value.status == bst.ERR_TIMEOUT
    w = wl.dense16(300, 200, 192, "f16", seed=11)
    got = run_dense(w, "f16", bst.sched(2, 0))
    assert_close_f16(got, oracle_dense(w, "f16"))
    torch.cuda.synchronize()


def test_wait_check_rejects_limits_out_of_range():
    for ns in (0, 10_000_000_001):
        with pytest.raises(bst.BstError) as e:
            bst.wait_check(ns, arrive=False)
        assert e.value.status == bst.ERR_INVALID_ARG
    bst.check_async()
