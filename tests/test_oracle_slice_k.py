"""Pins for the grouped slice-K oracle (05_grouped_matmul_slice_k and
11_grouped_matmul_slice_k_per_token_dequant of "Block Dispatch Policies"):
exact rational and Python-integer brute force with ragged and empty groups,
the partition of K (the unrounded group products add up to the full-K
product), the one-group case, and planted slice mistakes these checks catch."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, gemm as og
from block_swizzled_tile_gb300 import workloads as wl


def _offsets(gk):
    return np.concatenate([[0], np.cumsum(gk)]).astype(int)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_slice_k_bruteforce_rationals_ragged_and_empty(dtype):
    g = np.random.default_rng(31)
    gk = [3, 0, 1, 5, 0, 2]
    K, M, N = sum(gk), 3, 4
    a = og.decode(wl.uniform16((M, K), -2, 2, dtype, wl._gen(g.integers(1 << 30))), dtype)
    b = og.decode(wl.uniform16((K, N), -2, 2, dtype, wl._gen(g.integers(1 << 30))), dtype)
    got = og.gemm_grouped_slice_k(a, b, gk, "f32")
    off = _offsets(gk)
    assert got.shape == (len(gk), M, N)
    for gi in range(len(gk)):
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(off[gi], off[gi + 1]))
                x = float(exact)
                assert Fraction(x) == exact
                assert got[gi, i, j] == np.float32(x)
    # empty groups give zero matrices
    assert not got[1].any() and not got[4].any()


def test_slice_k_groups_partition_k():
    """The K slices partition [0, K): the unrounded group products add up to
    the full-K product, and each equals the product of its own slice."""
    g = np.random.default_rng(32)
    gk = [7, 1, 0, 12, 4]
    K = sum(gk)
    a = g.standard_normal((5, K))
    b = g.standard_normal((K, 6))
    parts = og.gemm_grouped_slice_k_f64(a, b, gk)
    np.testing.assert_allclose(parts.sum(axis=0), a @ b, rtol=0, atol=1e-12)
    off = _offsets(gk)
    np.testing.assert_allclose(parts[3], a[:, off[3]:off[4]] @ b[off[3]:off[4]], rtol=0, atol=1e-12)


def test_slice_k_single_group_is_plain():
    g = wl._gen(33)
    a = og.decode(wl.uniform16((9, 40), -1, 1, "bf16", g), "bf16")
    b = og.decode(wl.uniform16((40, 7), -1, 1, "bf16", g), "bf16")
    got = og.gemm_grouped_slice_k(a, b, [40], "bf16")
    assert np.array_equal(got[0], og.gemm(a, b, "bf16"))


def test_slice_k_rejects_bad_sizes():
    a = np.ones((2, 5))
    b = np.ones((5, 3))
    with pytest.raises(ValueError):
        og.gemm_grouped_slice_k(a, b, [2, 2], "f32")
    with pytest.raises(ValueError):
        og.gemm_grouped_slice_k(a, b, [6, -1], "f32")


def test_slice_k_quant_bruteforce_and_scales():
    """Python-integer brute force; each group uses its own row and column
    scales, and doubling one group's row scale doubles exactly that group's
    row."""
    g = wl._gen(34)
    gk = [4, 0, 6, 1]
    K, M, N = sum(gk), 3, 5
    a = wl.uniform_int8((M, K), g)
    b = wl.uniform_int8((K, N), g)
    sa = np.array([[1, 2, 4], [8, 8, 8], [0.5, 0.25, 2], [1, 1, 1]], np.float32)
    sb = np.array([[1, 2, 4, 8, 16], [1] * 5, [2, 2, 0.5, 1, 4], [0.125, 1, 1, 1, 1]], np.float32)
    acc, out = og.gemm_grouped_slice_k_quant_per_token(a, b, gk, sa, sb)
    off = _offsets(gk)
    for gi in range(len(gk)):
        for i in range(M):
            for j in range(N):
                want = sum(int(a[i, k]) * int(b[k, j]) for k in range(off[gi], off[gi + 1]))
                assert acc[gi, i, j] == want
                assert out[gi, i, j] == formats.f64_to_bf16_bits(
                    np.array([want * float(sa[gi, i]) * float(sb[gi, j])]))[0]
    sa2 = sa.copy()
    sa2[2, 1] *= 2
    _, out2 = og.gemm_grouped_slice_k_quant_per_token(a, b, gk, sa2, sb)
    changed = np.argwhere(out2 != out)
    assert changed.size and set(map(tuple, changed[:, :2])) <= {(2, 1)}
    assert np.array_equal(formats.bf16_bits_to_f64(out2[2, 1]), 2 * formats.bf16_bits_to_f64(out[2, 1]))


def test_slice_k_quant_single_group_is_plain_quant():
    g = wl._gen(35)
    a = wl.uniform_int8((6, 30), g)
    b = wl.uniform_int8((30, 4), g)
    sa = wl.uniform_f32((6,), 1e-3, 1e-2, g)
    sb = wl.uniform_f32((4,), 1e-3, 1e-2, g)
    acc1, out1 = og.gemm_quant_per_token(a, b, sa, sb)
    acc2, out2 = og.gemm_grouped_slice_k_quant_per_token(a, b, [30], sa[None], sb[None])
    assert np.array_equal(acc1, acc2[0]) and np.array_equal(out1, out2[0])


# ---- planted mistakes in the oracle must fail the pins above ---------------

def test_planted_slice_offset_is_caught(monkeypatch):
    """An oracle whose slices started one column late would no longer
    partition K: the partition pin sees it."""
    real = og._k_offsets

    def late(group_k, k_total):
        sizes, offs = real(group_k, k_total)
        return sizes, [0] + [min(o + 1, k_total) for o in offs[1:]]
    monkeypatch.setattr(og, "_k_offsets", late)
    g = np.random.default_rng(36)
    gk = [3, 4, 5]
    a = g.standard_normal((2, 12))
    b = g.standard_normal((12, 2))
    parts = og.gemm_grouped_slice_k_f64(a, b, gk)
    off = _offsets(gk)
    assert not np.allclose(parts[1], a[:, off[1]:off[2]] @ b[off[1]:off[2]], rtol=0, atol=1e-12)


def test_planted_dropped_group_is_caught(monkeypatch):
    """An oracle that skipped the last group would break the partition pin."""
    real = og.gemm_f64
    calls = []

    def skip_last(a, b):
        calls.append(1)
        return real(a, b) * (0.0 if len(calls) == 3 else 1.0)
    monkeypatch.setattr(og, "gemm_f64", skip_last)
    g = np.random.default_rng(37)
    a = g.standard_normal((3, 9))
    b = g.standard_normal((9, 3))
    parts = og.gemm_grouped_slice_k_f64(a, b, [2, 3, 4])
    assert not np.allclose(parts.sum(axis=0), a @ b, rtol=0, atol=1e-12)
