"""CPU oracle for the block-swizzled tile GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA path in ``block_swizzled_tile_gb300``.

What it computes, and where the definition comes from:

* ``oracle.swizzle`` -- the task-index -> output-tile mapping of
  ``GemmIdentityBlockSwizzle`` ("Block Scheduler Code Explained", sections
  4.3 GetCoreLoops, 4.4 GetBatchIdx, 4.5 GetBlockCoord, 4.6
  GetActualBlockShape, 5 Scheduling Policies, 6 Dynamic Scheduling
  Extension), in exact Python integers.
* ``oracle.formats`` -- decoders/encoders for fp16, bf16, float8 e4m3 and
  E8M0 written from the formats' definitions.
* ``oracle.gemm`` -- the plain definition of the contraction the method
  computes, C = A.B summed in fp64 (exact integers for int8), rounded once to
  the output type, for the plain, batched, grouped slice-M, MXFP8 and int8
  per-token-dequant variants named in "Block Dispatch Policies"
  (examples 00_basic_matmul, 01_batched_matmul, 02_grouped_matmul_slice_m,
  12_quant_matmul) and the MXFP8 GEMM of "MI450 WMMA and ds_load Scheduling
  via a DAG Mutation" ("An example run on a real kernel").

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force and library routines.  The Nz branch of GetBlockCoord
is elided on the page; the oracle's reading of it (the transpose of Zn) is
pinned by invariants and closed forms only -- see the docstring of
``oracle.swizzle.block_coord``.
"""
from . import formats, swizzle, gemm  # noqa: F401
