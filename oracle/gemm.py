"""The contraction the swizzled-tile GEMM computes, by its plain definition.
TEST INFRASTRUCTURE ONLY.

The scheduler of "Block Scheduler Code Explained" only reorders which tile is
computed when (sections 4.5-4.6, 7); the buffered mainloops of "Block Dispatch
Policies" only overlap loads with MMAs.  Neither changes the result, so the
result has a plain definition:

    C[i, j] = round_out( sum_k A[i, k] * B[k, j] )

summed in float64 (exact integers for int8) and rounded once, to nearest even,
to the output type.  The fp64 product uses numpy's matmul as a library
primitive; there is no blocking, fusion or reordering of our own.

Variants, as the example list of "Block Dispatch Policies" names them:
* ``gemm``          00_basic_matmul
* ``gemm_batched``  01_batched_matmul (GetBatchIdx of "Block Scheduler Code
                    Explained" section 4.4 splits tasks into batches)
* ``gemm_grouped``  02_grouped_matmul_slice_m: consecutive row slices of A and
                    C, one B per group
* ``gemm_quant_per_token`` 12_quant_matmul /
                    10_grouped_matmul_slice_m_per_token_dequant: int8 operands,
                    int32 accumulators, one fp32 scale per row of A (the
                    "token") and one per column of B.
* ``gemm_grouped_slice_k`` 05_grouped_matmul_slice_k: consecutive column
                    slices of A times the matching row slices of B, one output
                    matrix per group
* ``gemm_grouped_slice_k_quant_per_token``
                    11_grouped_matmul_slice_k_per_token_dequant: the same
                    slices on int8 operands with each group dequantised by its
                    own per-row and per-column scales
* ``gemm_mxfp8``    the MXFP8 GEMM of "MI450 WMMA and ds_load Scheduling via a
                    DAG Mutation" (float8 e4m3 A and B with one E8M0 scale per
                    32 consecutive K elements of each row of A and column of B).

Matrices enter in logical orientation: ``a`` is [M, K] and ``b`` is [K, N]
(``as_logical`` turns row- or column-major storage with a leading dimension
into that view).
"""
import numpy as np

from . import formats

_EXACT_INT_LIMIT = 2.0 ** 53   # every integer below this is exact in float64


def as_logical(storage, rows, cols, ld, col_major):
    """View a flat buffer as the logical [rows, cols] matrix.

    Row-major: element (r, c) sits at r*ld + c.  Column-major: at c*ld + r."""
    flat = np.asarray(storage).reshape(-1)
    if col_major:
        return np.lib.stride_tricks.as_strided(
            flat, shape=(rows, cols), strides=(flat.itemsize, ld * flat.itemsize))
    return np.lib.stride_tricks.as_strided(
        flat, shape=(rows, cols), strides=(ld * flat.itemsize, flat.itemsize))


def round_out(acc, out_dtype):
    """Round a float64 result once to the output type; returns raw storage
    (uint16 bits for 'f16'/'bf16', float32 values for 'f32')."""
    if out_dtype == "f16":
        return formats.f64_to_f16_bits(acc)
    if out_dtype == "bf16":
        return formats.f64_to_bf16_bits(acc)
    if out_dtype == "f32":
        return formats.f64_to_f32(acc)
    raise ValueError(out_dtype)


def decode(storage, dtype):
    """Raw operand storage -> float64 values."""
    if dtype == "f16":
        return formats.f16_bits_to_f64(storage)
    if dtype == "bf16":
        return formats.bf16_bits_to_f64(storage)
    if dtype == "e4m3":
        return formats.decode_e4m3(storage)
    if dtype == "s8":
        return np.asarray(storage, dtype=np.int8).astype(np.float64)
    if dtype == "f32":
        return np.asarray(storage, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def gemm_f64(a, b):
    """sum_k a[i,k] * b[k,j] in float64 (no rounding to the output yet)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape[1] != b.shape[0]:
        raise ValueError("inner dimensions differ")
    if a.shape[1] == 0:
        return np.zeros((a.shape[0], b.shape[1]))
    return a @ b


def gemm(a, b, out_dtype):
    """00_basic_matmul: C = round_out(A.B) with A [M,K], B [K,N] in float64."""
    return round_out(gemm_f64(a, b), out_dtype)


def gemm_batched(a, b, out_dtype):
    """01_batched_matmul: a [batch, M, K], b [batch, K, N]; each batch is an
    independent ``gemm``."""
    return np.stack([gemm(a[i], b[i], out_dtype) for i in range(a.shape[0])])


def gemm_grouped(x, w, group_m, out_dtype):
    """02_grouped_matmul_slice_m: rows [off_g, off_g + M_g) of x and of the
    output use weight w[g]; off_g is the sum of the earlier group sizes.
    Groups of size 0 contribute no rows.  x is [sum M_g, K], w is [G, K, N]."""
    x = np.asarray(x, dtype=np.float64)
    total = int(sum(group_m))
    if total != x.shape[0]:
        raise ValueError("group sizes do not add up to the rows of x")
    parts = []
    off = 0
    for g, mg in enumerate(group_m):
        parts.append(gemm(x[off:off + mg], w[g], out_dtype))
        off += mg
    return np.concatenate(parts, axis=0)


def mx_dequant_operand(codes, scales, block=32):
    """Element (r, k) of an MX operand is e4m3(codes[r, k]) * 2**(scales[r, k//32]-127)."""
    vals = formats.decode_e4m3(codes)
    sc = formats.decode_e8m0(scales)
    if vals.shape[1] != sc.shape[1] * block:
        raise ValueError("need one scale per %d K elements" % block)
    return vals * np.repeat(sc, block, axis=1)


def gemm_mxfp8(a_codes, a_scales, b_codes, b_scales, out_dtype="bf16"):
    """MXFP8 GEMM.  a_codes [M, K] and b_codes [N, K] hold e4m3 codes of the
    rows of A and of the columns of B (both K-contiguous); a_scales [M, K/32]
    and b_scales [N, K/32] hold E8M0 codes.  Products of e4m3 values and
    powers of two are exact in float64; the sum is taken in float64 and
    rounded once."""
    a = mx_dequant_operand(a_codes, a_scales)
    b = mx_dequant_operand(b_codes, b_scales)
    return round_out(gemm_f64(a, b.T), out_dtype)


def int_gemm_exact(a, b):
    """sum_k a[i,k]*b[k,j] for integer matrices, exactly, as int64.

    Computed with a float64 matmul: each product and every partial sum is an
    integer whose magnitude is at most K * max|a| * max|b|; below 2**53 every
    such integer is exact in float64, so any summation order gives the exact
    sum.  The bound is checked before multiplying."""
    a = np.asarray(a)
    b = np.asarray(b)
    K = a.shape[1]
    amax = float(np.abs(a.astype(np.int64)).max()) if a.size else 0.0
    bmax = float(np.abs(b.astype(np.int64)).max()) if b.size else 0.0
    if K * amax * bmax >= _EXACT_INT_LIMIT:
        raise ValueError("sum could exceed 2**53; float64 would not be exact")
    return gemm_f64(a.astype(np.float64), b.astype(np.float64)).astype(np.int64)


def gemm_quant_per_token(a, b, scale_a, scale_b, out_dtype="bf16"):
    """12_quant_matmul with per-token dequant.

    a [M, K] int8, b [K, N] int8 (logical), scale_a [M] and scale_b [N] fp32.
    acc[i, j] = sum_k a[i,k] * b[k,j] exactly (it must fit int32);
    C[i, j] = round_out(acc[i, j] * scale_a[i] * scale_b[j]) with the
    products in float64.  Returns (acc as int32, C)."""
    acc = int_gemm_exact(a, b)
    if acc.size and (acc.max() > 2**31 - 1 or acc.min() < -2**31):
        raise ValueError("accumulator does not fit int32")
    sa = np.asarray(scale_a, dtype=np.float32).astype(np.float64)
    sb = np.asarray(scale_b, dtype=np.float32).astype(np.float64)
    out = acc.astype(np.float64) * sa[:, None] * sb[None, :]
    return acc.astype(np.int32), round_out(out, out_dtype)


def gemm_grouped_quant_per_token(a, b, group_m, scale_a, scale_b, out_dtype="bf16"):
    """10_grouped_matmul_slice_m_per_token_dequant: the row slices of
    02_grouped_matmul_slice_m combined with the per-token dequant of
    12_quant_matmul.  Rows [off_g, off_g + M_g) of a (int8 [sum M_g, K]) use
    b[g] (int8 [K, N], logical) and scale_b[g] ([N]); scale_a holds one scale
    per row of a.  acc[i, j] = sum_k a[i,k] * b[g][k,j] exactly;
    C[i, j] = round_out(acc[i, j] * scale_a[i] * scale_b[g][j]) with the
    products in float64.  Returns (acc as int32, C)."""
    a = np.asarray(a)
    total = int(sum(group_m))
    if total != a.shape[0]:
        raise ValueError("group sizes do not add up to the rows of a")
    n = np.asarray(b[0]).shape[1] if len(b) else 0
    acc = np.zeros((total, n), dtype=np.int64)
    out = np.zeros((total, n), dtype=np.float64)
    sa = np.asarray(scale_a, dtype=np.float32).astype(np.float64)
    off = 0
    for g, mg in enumerate(group_m):
        if mg:
            acc_g = int_gemm_exact(a[off:off + mg], b[g])
            sb = np.asarray(scale_b[g], dtype=np.float32).astype(np.float64)
            acc[off:off + mg] = acc_g
            out[off:off + mg] = acc_g.astype(np.float64) * sa[off:off + mg, None] * sb[None, :]
        off += mg
    if acc.size and (acc.max() > 2**31 - 1 or acc.min() < -2**31):
        raise ValueError("accumulator does not fit int32")
    return acc.astype(np.int32), round_out(out, out_dtype)


def _k_offsets(group_k, k_total):
    """Exclusive prefix sums of the group K sizes; they must cover exactly
    k_total columns of A (rows of B)."""
    sizes = [int(k) for k in group_k]
    if any(k < 0 for k in sizes):
        raise ValueError("negative group size")
    if sum(sizes) != k_total:
        raise ValueError("group sizes do not add up to K")
    offs = [0]
    for k in sizes:
        offs.append(offs[-1] + k)
    return sizes, offs


def gemm_grouped_slice_k_f64(a, b, group_k):
    """The unrounded products of 05_grouped_matmul_slice_k: for group g with
    K slice [off_g, off_g + K_g), part[g] = sum over k in the slice of
    a[i, k] * b[k, j] in float64.  a is [M, sum K_g], b is [sum K_g, N];
    returns [G, M, N].  A group with K_g = 0 gives a zero matrix."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    sizes, offs = _k_offsets(group_k, a.shape[1])
    if b.shape[0] != a.shape[1]:
        raise ValueError("inner dimensions differ")
    out = np.zeros((len(sizes), a.shape[0], b.shape[1]), dtype=np.float64)
    for g, kg in enumerate(sizes):
        if kg:
            out[g] = gemm_f64(a[:, offs[g]:offs[g + 1]], b[offs[g]:offs[g + 1], :])
    return out


def gemm_grouped_slice_k(a, b, group_k, out_dtype):
    """05_grouped_matmul_slice_k: C[g] = round_out(A[:, slice g] . B[slice g, :]),
    each group's float64 sum rounded once."""
    return round_out(gemm_grouped_slice_k_f64(a, b, group_k), out_dtype)


def gemm_grouped_slice_k_quant_per_token(a, b, group_k, scale_a, scale_b, out_dtype="bf16"):
    """11_grouped_matmul_slice_k_per_token_dequant: the K slices of
    05_grouped_matmul_slice_k on int8 a [M, sum K_g] and b [sum K_g, N]
    (logical), each group dequantised as 12_quant_matmul does:
    acc[g][i, j] = sum over k in slice g of a[i,k] * b[k,j] exactly (it must
    fit int32), C[g][i, j] = round_out(acc[g][i, j] * scale_a[g][i] *
    scale_b[g][j]) with the products in float64.  scale_a is [G, M] and
    scale_b [G, N].  Returns (acc as int32 [G, M, N], C)."""
    a = np.asarray(a)
    b = np.asarray(b)
    sizes, offs = _k_offsets(group_k, a.shape[1])
    G, M, N = len(sizes), a.shape[0], b.shape[1]
    acc = np.zeros((G, M, N), dtype=np.int64)
    for g, kg in enumerate(sizes):
        if kg:
            acc[g] = int_gemm_exact(a[:, offs[g]:offs[g + 1]], b[offs[g]:offs[g + 1], :])
    if acc.size and (acc.max() > 2**31 - 1 or acc.min() < -2**31):
        raise ValueError("accumulator does not fit int32")
    sa = np.asarray(scale_a, dtype=np.float32).astype(np.float64).reshape(G, M)
    sb = np.asarray(scale_b, dtype=np.float32).astype(np.float64).reshape(G, N)
    out = acc.astype(np.float64) * sa[:, :, None] * sb[:, None, :]
    return acc.astype(np.int32), round_out(out, out_dtype)
