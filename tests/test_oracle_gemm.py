"""Pins for oracle.gemm: exact rational brute force on tiny problems, a
textbook product, special cases (identity, zero, K = 0), closed forms for the
grouped, batched, MXFP8 and per-token-dequant variants, exact integer sums,
and planted mistakes that these checks must catch."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, gemm as og
from block_swizzled_tile_gb300 import workloads as wl


def _exact_round(values, out_dtype):
    """Round exact rationals through the brute-force-pinned encoder: a
    Fraction is first made a float64 only where that is exact (tiny sums of
    fp16 products are), which the asserts below check."""
    f = np.array([float(v) for v in values])
    for v, x in zip(values, f):
        assert Fraction(x) == v, "tiny case must be exact in float64"
    return og.round_out(f, out_dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out", ["f16", "bf16", "f32"])
def test_bruteforce_rationals(dtype, out):
    g = np.random.default_rng(5)
    for M, N, K in [(1, 1, 1), (3, 2, 5), (4, 4, 7), (2, 5, 3)]:
        a_bits = wl.uniform16((M, K), -2, 2, dtype, wl._gen(g.integers(1 << 30)))
        b_bits = wl.uniform16((K, N), -2, 2, dtype, wl._gen(g.integers(1 << 30)))
        a = og.decode(a_bits, dtype)
        b = og.decode(b_bits, dtype)
        exact = [sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K))
                 for i in range(M) for j in range(N)]
        want = _exact_round(exact, out).reshape(M, N)
        got = og.gemm(a, b, out)
        assert np.array_equal(got, want)


def test_textbook_product():
    a = np.array([[1.0, 2.0], [3.0, 4.0]])
    b = np.array([[5.0, 6.0], [7.0, 8.0]])
    got = formats.f16_bits_to_f64(og.gemm(a, b, "f16"))
    assert np.array_equal(got, [[19, 22], [43, 50]])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_and_zero(dtype):
    w = wl.dense16(37, 37, 37, dtype, seed=3)
    a = og.decode(w["a"], dtype)
    eye = np.eye(37)
    assert np.array_equal(og.gemm(a, eye, dtype), w["a"])   # same format out: exact
    assert not og.gemm(a, np.zeros((37, 5)), "f32").any()
    assert og.gemm(np.zeros((4, 0)), np.zeros((0, 6)), "f16").shape == (4, 6)
    assert not formats.f16_bits_to_f64(og.gemm(np.zeros((4, 0)), np.zeros((0, 6)), "f16")).any()


def test_as_logical_layouts():
    flat = np.arange(3 * 7, dtype=np.uint16)
    rm = og.as_logical(flat, 3, 5, 7, col_major=False)       # ld 7 > cols 5
    assert np.array_equal(rm, flat.reshape(3, 7)[:, :5])
    cm = og.as_logical(flat, 5, 3, 7, col_major=True)
    assert np.array_equal(cm, flat.reshape(3, 7)[:, :5].T)


def test_batched_closed_form():
    """Batch i multiplies its own A_i by B_i = (i+1) * I, so output batch i is
    (i+1) * A_i rounded once; a mixed-up batch index or a shared operand
    fails it."""
    batch, M, K = 4, 9, 12
    g = wl._gen(31)
    a = np.stack([og.decode(wl.uniform16((M, K), -1, 1, "bf16", g), "bf16") for _ in range(batch)])
    b = np.stack([(i + 1) * np.eye(K) for i in range(batch)])
    got = formats.bf16_bits_to_f64(og.gemm_batched(a, b, "bf16"))
    for i in range(batch):
        want = formats.bf16_bits_to_f64(formats.f64_to_bf16_bits((i + 1) * a[i]))
        assert np.array_equal(got[i], want)
    assert not np.array_equal(got[0], got[1])


def _triple_loop_f64(a, b):
    """sum_k a[i,k]*b[k,j] by an explicit loop over i, j, k in float64."""
    M, K = a.shape
    N = b.shape[1]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += float(a[i, k]) * float(b[k, j])
            out[i, j] = s
    return out


def _triple_loop_int(a, b):
    M, K = a.shape
    N = b.shape[1]
    return [[sum(int(a[i, k]) * int(b[k, j]) for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matmul_primitive_agrees_with_triple_loop(dtype):
    """The oracle's float64 product uses numpy's matmul as a library
    primitive; an explicit triple loop (the plain definition) must give the
    same sums.  The two differ only in summation order, so they agree to
    float64 rounding, and after the one rounding to the output type they
    are identical on these shapes."""
    g = wl._gen(32)
    for M, N, K in [(1, 1, 1), (3, 4, 5), (7, 5, 33), (16, 9, 70), (2, 3, 0)]:
        a = og.decode(wl.uniform16((M, K), -1, 1, dtype, g), dtype)
        b = og.decode(wl.uniform16((K, N), -1, 1, dtype, g), dtype)
        loop = _triple_loop_f64(a, b)
        prim = og.gemm_f64(a, b)
        assert np.allclose(prim, loop, rtol=1e-14, atol=1e-300)
        assert np.array_equal(og.round_out(loop, dtype), og.gemm(a, b, dtype))


def test_int_primitive_agrees_with_triple_loop():
    g = wl._gen(33)
    for M, N, K in [(4, 3, 1), (6, 5, 17), (3, 7, 129)]:
        a = wl.uniform_int8((M, K), g)
        b = wl.uniform_int8((K, N), g)
        assert og.int_gemm_exact(a, b).tolist() == _triple_loop_int(a, b)
        acc, _ = og.gemm_quant_per_token(a, b, np.ones(M, np.float32), np.ones(N, np.float32))
        assert acc.tolist() == _triple_loop_int(a, b)


def test_grouped_closed_form():
    # weight of group g is (g+1) * I, so output rows of group g are (g+1) * x
    gm = [3, 0, 5, 1, 0, 2]
    K = N = 8
    x = og.decode(wl.uniform16((sum(gm), K), -1, 1, "bf16", wl._gen(4)), "bf16")
    w = np.stack([(g + 1) * np.eye(K) for g in range(len(gm))])
    got = formats.bf16_bits_to_f64(og.gemm_grouped(x, w, gm, "bf16"))
    scale = np.repeat([g + 1 for g in range(len(gm))], gm)[:, None]
    assert np.array_equal(got, formats.bf16_bits_to_f64(formats.f64_to_bf16_bits(x * scale)))


def test_grouped_single_group_is_plain():
    w = wl.grouped_bf16(group_m=[50], N=24, K=40, seed=2)
    x = og.decode(w["x"], "bf16")
    ww = og.decode(w["w"], "bf16")
    assert np.array_equal(og.gemm_grouped(x, ww, [50], "bf16"), og.gemm(x, ww[0], "bf16"))


def test_grouped_rejects_bad_sizes():
    with pytest.raises(ValueError):
        og.gemm_grouped(np.zeros((5, 2)), np.zeros((2, 2, 2)), [2, 2], "bf16")


def test_mxfp8_unit_scales_reduce_to_plain_e4m3():
    w = wl.mxfp8(M=16, N=24, K=96, seed=7)
    ones_a = np.full_like(w["sa"], 127)
    ones_b = np.full_like(w["sb"], 127)
    got = og.gemm_mxfp8(w["a"], ones_a, w["b"], ones_b)
    plain = og.gemm(formats.decode_e4m3(w["a"]), formats.decode_e4m3(w["b"]).T, "bf16")
    assert np.array_equal(got, plain)


def test_mxfp8_scale_block_doubles_its_contribution():
    w = wl.mxfp8(M=8, N=8, K=96, seed=8)
    a = formats.decode_e4m3(w["a"])
    b = formats.decode_e4m3(w["b"])
    sa = w["sa"].copy()
    i, kb = 3, 1
    sa2 = sa.copy()
    sa2[i, kb] += 1
    base = og.gemm_f64(og.mx_dequant_operand(w["a"], sa), og.mx_dequant_operand(w["b"], w["sb"]).T)
    bump = og.gemm_f64(og.mx_dequant_operand(w["a"], sa2), og.mx_dequant_operand(w["b"], w["sb"]).T)
    ks = slice(32 * kb, 32 * kb + 32)
    sa_row = formats.decode_e8m0(sa[i, kb])
    sb_blk = formats.decode_e8m0(w["sb"][:, kb])
    contrib = (a[i, ks] * sa_row) @ (b[:, ks] * sb_blk[:, None]).T
    diff = bump - base
    assert np.allclose(diff[i], contrib, rtol=0, atol=1e-9 * np.abs(base).max())
    others = np.delete(diff, i, axis=0)
    assert not others.any()


def test_int_exact_vs_python_ints():
    g = wl._gen(9)
    a = wl.uniform_int8((5, 11), g)
    b = wl.uniform_int8((11, 4), g)
    want = [[sum(int(a[i, k]) * int(b[k, j]) for k in range(11)) for j in range(4)] for i in range(5)]
    assert og.int_gemm_exact(a, b).tolist() == want


def test_int_exact_vs_int64_matmul_and_extreme():
    g = wl._gen(10)
    a = wl.uniform_int8((64, 777), g)
    b = wl.uniform_int8((777, 48), g)
    assert np.array_equal(og.int_gemm_exact(a, b), a.astype(np.int64) @ b.astype(np.int64))
    full = np.full((2, 8192), 127, np.int8)
    acc = og.int_gemm_exact(full, full.T)
    assert (acc == 8192 * 127 * 127).all()
    neg = np.full((1, 8192), -127, np.int8)
    assert og.int_gemm_exact(neg, full.T)[0, 0] == -8192 * 127 * 127


def test_quant_unit_scales_is_rounded_acc():
    g = wl._gen(11)
    a = wl.uniform_int8((9, 64), g)
    b = wl.uniform_int8((64, 7), g)
    acc, out = og.gemm_quant_per_token(a, b, np.ones(9, np.float32), np.ones(7, np.float32))
    assert np.array_equal(out, formats.f64_to_bf16_bits(acc.astype(np.float64)))


def test_quant_scales_are_row_and_column():
    g = wl._gen(12)
    a = wl.uniform_int8((6, 32), g)
    b = wl.uniform_int8((32, 5), g)
    sa = np.array([1, 2, 4, 8, 0.5, 0.25], np.float32)
    sb = np.array([1, 2, 4, 8, 16], np.float32)
    acc, out = og.gemm_quant_per_token(a, b, sa, sb)
    want = formats.f64_to_bf16_bits(acc * sa[:, None].astype(np.float64) * sb[None, :].astype(np.float64))
    assert np.array_equal(out, want)
    # powers of two scale exactly: row i of out is bf16(acc) scaled by sa[i]*sb[j]
    base = formats.bf16_bits_to_f64(formats.f64_to_bf16_bits(acc.astype(np.float64)))
    assert np.array_equal(formats.bf16_bits_to_f64(out), base * sa[:, None] * sb[None, :])


def test_grouped_quant_single_group_is_plain_quant():
    g = wl._gen(21)
    a = wl.uniform_int8((10, 48), g)
    b = wl.uniform_int8((48, 9), g)
    sa = wl.uniform_f32((10,), 1e-3, 1e-2, g)
    sb = wl.uniform_f32((9,), 1e-3, 1e-2, g)
    acc1, out1 = og.gemm_quant_per_token(a, b, sa, sb)
    acc2, out2 = og.gemm_grouped_quant_per_token(a, b[None], [10], sa, sb[None])
    assert np.array_equal(acc1, acc2) and np.array_equal(out1, out2)


def test_grouped_quant_brute_force_and_empty_groups():
    """Python-integer brute force on a tiny problem with empty groups; a
    power-of-two change of one group's column scale moves only that group's
    rows of that column."""
    g = wl._gen(22)
    gm = [2, 0, 3, 0, 1]
    K, N = 5, 4
    a = wl.uniform_int8((6, K), g)
    b = wl.uniform_int8((5, K, N), g)
    sa = np.array([1, 2, 4, 0.5, 8, 0.25], np.float32)
    sb = np.array([[1, 2, 4, 8]] * 5, np.float32)
    acc, out = og.gemm_grouped_quant_per_token(a, b, gm, sa, sb)
    off = np.concatenate([[0], np.cumsum(gm)])
    for gi in range(5):
        for i in range(off[gi], off[gi + 1]):
            for j in range(N):
                want = sum(int(a[i, k]) * int(b[gi][k, j]) for k in range(K))
                assert acc[i, j] == want
                assert out[i, j] == formats.f64_to_bf16_bits(np.array([want * float(sa[i]) * float(sb[gi][j])]))[0]
    sb2 = sb.copy()
    sb2[2, 1] *= 4
    acc2, out2 = og.gemm_grouped_quant_per_token(a, b, gm, sa, sb2)
    changed = out2 != out
    rows = set(np.nonzero(changed)[0]) | set()
    assert rows <= set(range(off[2], off[3])) and set(np.nonzero(changed)[1]) <= {1}
    assert np.array_equal(formats.bf16_bits_to_f64(out2[off[2]:off[3], 1]),
                          formats.bf16_bits_to_f64(out[off[2]:off[3], 1]) * 4)


# ---- planted mistakes in the oracle must fail the pins above ---------------

def test_planted_transpose_is_caught(monkeypatch):
    # an oracle that multiplied in the wrong order (B.A instead of A.B) must
    # fail the textbook pin: the textbook product does not commute
    real = og.gemm_f64
    monkeypatch.setattr(og, "gemm_f64", lambda a, b: real(b, a))
    a = np.array([[1.0, 2.0], [3.0, 4.0]])
    b = np.array([[5.0, 6.0], [7.0, 8.0]])
    got = formats.f16_bits_to_f64(og.gemm(a, b, "f16"))
    assert not np.array_equal(got, [[19, 22], [43, 50]])


def test_planted_wrong_group_weight_is_caught(monkeypatch):
    gm = [3, 0, 5, 1]
    K = N = 4
    x = np.ones((sum(gm), K))
    w = np.stack([(g + 1) * np.eye(K) for g in range(len(gm))])
    real = og.gemm_grouped

    def shifted(x, w, gm, out):       # uses the next group's weight
        return real(x, np.roll(w, -1, axis=0), gm, out)
    got = formats.bf16_bits_to_f64(shifted(x, w, gm, "bf16"))
    scale = np.repeat([g + 1 for g in range(len(gm))], gm)[:, None]
    assert not np.array_equal(got, x * scale)


def test_planted_scale_axis_mixup_is_caught():
    g = wl._gen(13)
    a = wl.uniform_int8((6, 32), g)
    b = wl.uniform_int8((32, 6), g)
    sa = np.array([1, 3, 2, 7, 5, 4], np.float32)
    sb = np.array([2, 1, 9, 4, 3, 8], np.float32)
    acc, out = og.gemm_quant_per_token(a, b, sa, sb)
    wrong = formats.f64_to_bf16_bits(acc * sb[:, None].astype(np.float64) * sa[None, :].astype(np.float64))
    assert not np.array_equal(out, wrong)
