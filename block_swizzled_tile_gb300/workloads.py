"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and packs them into the raw storage the
library consumes (fp16/bf16 bits as uint16, e4m3 and E8M0 codes as uint8,
int8, fp32).  It holds none of the GEMM's arithmetic; the tests, the bench and
the smoke check feed the same bytes to the CUDA path and to the CPU oracle.

Every workload is a plain dict of numpy arrays plus shape/layout fields:
``M, N, K``; ``a`` with ``lda``/``a_col_major``; ``b`` with ``ldb``/
``b_col_major`` where B is the logical [K, N] operand; extra keys per kind.

Named workloads (the shapes and distributions the method is measured on):

* ``fp16_tail``     fp16, M=500 N=380 K=256, A and B row-major, U[-1, 1]
* ``fp16_square``   fp16, M=N=1024 K=2048, A row-major, B column-major,
                    N(0,1)/sqrt(K)
* ``mxfp8``         e4m3 A [1024, 4096] and B^T [2048, 4096] (K-contiguous),
                    N(0,1) clipped to +-448 then cast to e4m3; E8M0 scales
                    127 + U{-4..4}, one per 32 K per row/column
* ``grouped_bf16``  G=8 groups whose sizes are a multinomial draw of 8192 rows
                    over 8 equally likely groups; X [8192, 4096] ~ N(0,1),
                    W [8, 4096, 4096] ~ N(0, 0.02) (N contiguous), bf16
* ``int8_per_token`` A int8 [8192, 8192] and B^T int8 [8192, 8192]
                    (K-contiguous) ~ U{-127..127}; fp32 scales ~ U[1e-3, 1e-2]
                    per row of A and per column of B
"""
import math

import numpy as np
import torch


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _bits16(t):
    """A torch fp16/bf16 CPU tensor -> numpy uint16 bits."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _codes8(t):
    return t.contiguous().view(torch.uint8).numpy()


# ------------------------------------------------------------- primitives ---

def uniform16(shape, lo, hi, dtype, gen):
    """U[lo, hi) rounded to fp16 ('f16') or bf16 ('bf16'); uint16 bits."""
    x = torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    return _bits16(x.to(torch.float16 if dtype == "f16" else torch.bfloat16))


def normal16(shape, std, dtype, gen):
    """N(0, std^2) rounded to fp16/bf16; uint16 bits."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32) * std
    return _bits16(x.to(torch.float16 if dtype == "f16" else torch.bfloat16))


def normal_e4m3(shape, gen):
    """N(0,1) clipped to +-448 and cast to float8 e4m3; uint8 codes."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32).clamp_(-448.0, 448.0)
    return _codes8(x.to(torch.float8_e4m3fn))


def e8m0_scales(shape, gen, lo=-4, hi=4):
    """E8M0 codes 127 + U{lo..hi}, i.e. scales 2**U{lo..hi}."""
    return (torch.randint(127 + lo, 127 + hi + 1, shape, generator=gen)
            .to(torch.uint8).numpy())


def uniform_int8(shape, gen, lo=-127, hi=127):
    return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int8).numpy()


def uniform_f32(shape, lo, hi, gen):
    return (torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo).numpy()


def multinomial_groups(total, groups, gen):
    """Group sizes: ``total`` draws over ``groups`` equally likely groups,
    counted per group (zero-size groups are possible)."""
    draws = torch.multinomial(torch.ones(groups), total, replacement=True, generator=gen)
    return [int(v) for v in torch.bincount(draws, minlength=groups).tolist()]


# ---------------------------------------------------------------- generic ---

def dense16(M, N, K, dtype="f16", a_col_major=False, b_col_major=False,
            dist="uniform", seed=0, lda=None, ldb=None, batch=1):
    """A generic fp16/bf16 problem.  A is [M, K], B is [K, N] (logical); a
    column-major operand is stored transposed.  ``lda``/``ldb`` default to the
    dense leading dimension; larger values pad each row (padding is random)."""
    g = _gen(seed)
    a_rows, a_cols = (K, M) if a_col_major else (M, K)
    b_rows, b_cols = (N, K) if b_col_major else (K, N)
    lda = a_cols if lda is None else lda
    ldb = b_cols if ldb is None else ldb

    def draw(rows, ld):
        shape = (batch, rows, ld) if batch > 1 else (rows, ld)
        if dist == "uniform":
            return uniform16(shape, -1.0, 1.0, dtype, g)
        return normal16(shape, 1.0 / math.sqrt(max(K, 1)), dtype, g)

    return dict(kind="dense", dtype=dtype, M=M, N=N, K=K, batch=batch,
                a=draw(a_rows, lda), lda=lda, a_col_major=a_col_major,
                b=draw(b_rows, ldb), ldb=ldb, b_col_major=b_col_major)


# ------------------------------------------------------------ named ones ---

def fp16_tail(seed=0):
    return dense16(500, 380, 256, "f16", a_col_major=False, b_col_major=False,
                   dist="uniform", seed=seed)


def fp16_square(seed=0):
    return dense16(1024, 1024, 2048, "f16", a_col_major=False, b_col_major=True,
                   dist="normal", seed=seed)


def mxfp8(M=1024, N=2048, K=4096, seed=0):
    g = _gen(seed)
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    return dict(kind="mxfp8", M=M, N=N, K=K,
                a=normal_e4m3((M, K), g), b=normal_e4m3((N, K), g),
                sa=e8m0_scales((M, K // 32), g), sb=e8m0_scales((N, K // 32), g))


def grouped_bf16(group_m=None, G=8, total_m=8192, N=4096, K=4096, seed=0):
    g = _gen(seed)
    if group_m is None:
        group_m = multinomial_groups(total_m, G, g)
    group_m = [int(v) for v in group_m]
    total = sum(group_m)
    return dict(kind="grouped", dtype="bf16", group_m=group_m, G=len(group_m), N=N, K=K,
                x=normal16((total, K), 1.0, "bf16", g),
                w=normal16((len(group_m), K, N), 0.02, "bf16", g))


def int8_per_token(M=8192, N=8192, K=8192, seed=0):
    g = _gen(seed)
    return dict(kind="int8", M=M, N=N, K=K,
                a=uniform_int8((M, K), g), b=uniform_int8((N, K), g),   # b is B^T: K contiguous
                sa=uniform_f32((M,), 1e-3, 1e-2, g), sb=uniform_f32((N,), 1e-3, 1e-2, g))


def grouped_int8_per_token(group_m=None, G=8, total_m=8192, N=4096, K=4096, seed=0):
    """Grouped slice-M int8 with per-token dequant: the group sizes of the
    grouped workload, the value distributions of the int8 one.  w holds each
    group's B^T ([G, N, K], K contiguous); sb one row of column scales per
    group."""
    g = _gen(seed)
    if group_m is None:
        group_m = multinomial_groups(total_m, G, g)
    group_m = [int(v) for v in group_m]
    total = sum(group_m)
    G = len(group_m)
    return dict(kind="grouped_int8", group_m=group_m, G=G, N=N, K=K,
                x=uniform_int8((total, K), g), w=uniform_int8((G, N, K), g),
                sa=uniform_f32((total,), 1e-3, 1e-2, g), sb=uniform_f32((G, N), 1e-3, 1e-2, g))


def grouped_slice_k_bf16(group_k=None, G=8, total_k=8192, M=4096, N=4096, seed=0):
    """Grouped slice-K, bf16: the token dimension is K and is split into G
    groups (sizes drawn like the grouped slice-M workload's), as in a weight
    gradient dW_g = X_g^T . dY_g.  x holds A^T ([sum K_g, M], M contiguous:
    A is MN-major) and dy holds B ([sum K_g, N], N contiguous: MN-major), both
    N(0, 1); the output is [G, M, N]."""
    g = _gen(seed)
    if group_k is None:
        group_k = multinomial_groups(total_k, G, g)
    group_k = [int(v) for v in group_k]
    total = sum(group_k)
    return dict(kind="slice_k", dtype="bf16", group_k=group_k, G=len(group_k), M=M, N=N,
                x=normal16((total, M), 1.0, "bf16", g), dy=normal16((total, N), 1.0, "bf16", g))


def grouped_slice_k_int8(group_k=None, G=8, total_k=8192, M=4096, N=4096, seed=0):
    """Grouped slice-K int8 with per-token dequant: the group sizes of the
    slice-K workload, the value distributions of the int8 one.  a is the
    logical A [M, sum K_g] and b the logical B [sum K_g, N] (U{-127..127});
    sa [G, M] and sb [G, N] hold each group's row and column scales."""
    g = _gen(seed)
    if group_k is None:
        group_k = multinomial_groups(total_k, G, g)
    group_k = [int(v) for v in group_k]
    total = sum(group_k)
    G = len(group_k)
    return dict(kind="slice_k_int8", group_k=group_k, G=G, M=M, N=N,
                a=uniform_int8((M, total), g), b=uniform_int8((total, N), g),
                sa=uniform_f32((G, M), 1e-3, 1e-2, g), sb=uniform_f32((G, N), 1e-3, 1e-2, g))
