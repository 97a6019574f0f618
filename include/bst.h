/*
 * bst.h -- block-swizzled tile GEMM for GB300 (sm_103a), C ABI.
 *
 * What the library computes is the dense contraction C = A.B with fp32
 * accumulation, in the variants named in "Block Dispatch Policies" (CATLASS
 * docs: examples 00_basic_matmul, 01_batched_matmul,
 * 02_grouped_matmul_slice_m, 12_quant_matmul) and the MXFP8 GEMM of "MI450
 * WMMA and ds_load Scheduling via a DAG Mutation" ("An example run on a real
 * kernel").  Output tiles are handed to persistent CTAs in the order of
 * GemmIdentityBlockSwizzle ("Block Scheduler Code Explained", sections 4-7):
 * windows of SwizzleOffset tile-rows (Zn) or tile-columns (Nz), reversed on
 * odd windows, tail tiles cut by GetActualBlockShape.
 *
 * Conventions for every entry point:
 *  - Matrices are dense 2-D (or 3-D batched/grouped) arrays in DEVICE memory
 *    owned by the caller; the library never allocates, frees or keeps them.
 *    A is logically [M, K], B is logically [K, N], C is [M, N] row-major.
 *    bst_layout says how an operand is stored: BST_ROW_MAJOR means element
 *    (r, c) of the logical matrix is at r*ld + c, BST_COL_MAJOR at c*ld + r.
 *    Leading dimensions and strides are in ELEMENTS.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) of the CURRENT device.  An argument error
 *    returns before anything is enqueued.  Device-side failures (a bounded
 *    wait that gave up, inconsistent group sizes) are recorded in a per-device
 *    error word and reported by bst_check_async.
 *  - Operands whose base address and leading dimension are 16-byte aligned
 *    are fetched with TMA.  A row-major fp16/bf16 B whose pitch is 8 bytes
 *    off a multiple of 16 (plain GEMMs, even K) is fetched with TMA through
 *    a view of pairs of its rows; other operands with ordinary loads
 *    (slower, same results).  There is no CPU fallback: without a usable
 *    sm_103a device the call returns BST_ERR_CUDA.
 *  - Environment switches, read once per process (for measurement; the
 *    results do not change): BST_PDL=0 launches without programmatic
 *    dependent launch; BST_PREFETCH_MB=n sets the operand size up to which
 *    a kernel pulls its operands into L2 at start (default 32, 0 = never);
 *    BST_ROWS2=0 turns the two-row view of B off; BST_WIDEN_BULK=0 widens
 *    int8 operands with ordinary loads instead of bulk copies.
 *  - Empty outputs (M == 0 or N == 0) return BST_OK without a launch; K == 0
 *    writes zeros.
 *  - The library holds no mutable host state except cached device properties,
 *    so calls from several host threads are safe.
 */
#ifndef BST_H
#define BST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BST_OK = 0,
    BST_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, ...   */
    BST_ERR_UNSUPPORTED = 2,   /* a dtype/layout combination not implemented   */
    BST_ERR_ALIGNMENT = 3,     /* an address or stride the path cannot take   */
    BST_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed            */
    BST_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up           */
    BST_ERR_DEVICE = 6         /* a device-side consistency check failed       */
} bst_status;

typedef enum {
    BST_F16 = 0,   /* IEEE binary16                                  */
    BST_BF16 = 1,  /* bfloat16                                       */
    BST_E4M3 = 2,  /* float8 e4m3 ("fn": no infinities, 0x7F NaN)    */
    BST_S8 = 3,    /* int8                                           */
    BST_F32 = 4,   /* IEEE binary32                                  */
    BST_S32 = 5    /* int32                                          */
} bst_dtype;

typedef enum { BST_ROW_MAJOR = 0, BST_COL_MAJOR = 1 } bst_layout;

/*
 * Scheduling parameters ("Block Scheduler Code Explained" section 2.1 and
 * section 6, DynamicGemmIdentityBlockSwizzle::SetSwizzleParams).  A NULL
 * bst_sched* means: offset 1, Zn, automatic tile and grid.
 */
typedef struct {
    uint32_t swizzle_offset;    /* SwizzleOffset, >= 1 (0 is rejected)                 */
    uint32_t swizzle_direction; /* SwizzleDirection: 0 = Zn, 1 = Nz                    */
    uint32_t tile_n;            /* 0 = automatic, else 64, 128 or 256                   */
    uint32_t tile_m;            /* 0 = automatic, 128 (one CTA per tile) or 256 (a pair
                                   of CTAs on one TPC per tile, tcgen05 cta_group::2;
                                   fp16/bf16 with 16-byte-aligned operands, tile_n 128
                                   or 256)                                             */
    uint32_t num_ctas;          /* persistent CTAs; 0 = one per SM                      */
    uint32_t split_k;           /* 0 = automatic, 1 = off, 2 or 4: each output tile
                                   is computed by 2 or 4 CTAs (or CTA pairs) over
                                   disjoint K ranges and summed through distributed
                                   shared memory.  Plain GEMMs only.  fp16/bf16 with
                                   16-byte-aligned operands: CTA pairs, tiles 256 x 256
                                   or 256 x 128.  fp16/bf16 with an operand TMA cannot
                                   fetch: single CTAs, tiles 128 x 64 (2 splits) or
                                   128 x 128 (2 or 4).  MXFP8: single CTAs, tiles
                                   128 x 256 (2 splits) or 128 x 128.  The automatic
                                   choice splits when the tiles alone leave SMs idle.
                                   The K ranges differ in size by at most one k-block;
                                   a range left empty (fewer k-blocks than splits)
                                   contributes zeros                                   */
    uint32_t* trace;            /* optional DEVICE buffer of 5 uint32 per task; when
                                   non-NULL the kernel writes, for task index t, the
                                   tile it computed: {batch or group, m, n, mActual,
                                   nActual}.  For grouped calls it must hold
                                   (ceil(total_m/128) + G) * ceil(N/tile_n) tasks.
                                   Debug only.                                        */
    uint64_t* timeline;         /* optional DEVICE buffer of 64 uint64 per CTA (row =
                                   block index); when non-NULL the GEMM kernels write
                                   %globaltimer stamps (ns) of their pipeline events.
                                   Persistent kernels: [0] set-up done (after the
                                   grid-dependency wait), [1..15] A-load issues of the
                                   first k-blocks, [8..14] copy or two-row-view B
                                   batches, [16..31] MMA k-block starts, [32..39] /
                                   [40..47] epilogue tile starts / ends, [48..50] exit
                                   of warps 0, 1, 2; one-CTA kernels also [55] entry and
                                   [56] / [57] before / after the first tile's
                                   coordinates; the MXFP8 pair kernel instead has [0]
                                   entry, [53] / [52] after the wait / the dependent-
                                   launch trigger, [54] first load, [56..61] scale
                                   groups rewritten.  Split-K pair kernels: [0] entry,
                                   [44] after the wait, [1] after the trigger, [2..15]
                                   A-load issues, [16..31] MMA k-block starts, [32]
                                   accumulator ready, [34] / [33] partials sent /
                                   received, per epilogue warp [48..51] partials
                                   received and [40..43] stores done, [36] epilogue done,
                                   [39] / [37] cluster barrier passed / TMEM freed.
                                   Profiling only (bench.py --timeline prints them).   */
    uint32_t shuffle_k;         /* 1: ShuffleK ("Block Dispatch Policies",
                                   ENABLE_SHUFFLE_K): the K loop of task t starts at
                                   k-block t % (k-blocks of the tile) and wraps, so
                                   tiles running at the same time read different
                                   k-blocks of a shared operand panel.  Changes only
                                   the fp32 summation order.  fp16/bf16 and int8
                                   paths (a split-K tile rotates within its split's
                                   K range, starting at (task + split) % its
                                   k-blocks); MXFP8 returns BST_ERR_UNSUPPORTED.     */
    uint32_t dynamic;           /* 1: dynamic task allocation ("Block Scheduler Code
                                   Explained" section 1): the grid holds one CTA-pair
                                   cluster per task; a cluster computes its own task,
                                   then claims the tasks of clusters that have not
                                   started, by hardware cluster launch control, until
                                   none is left.  Tasks keep their numbering (the
                                   trace is unchanged); which CTA runs which task is
                                   decided at run time.  CTA-pair tiles only
                                   (tile_m 256 is implied; 128 is
                                   BST_ERR_UNSUPPORTED); num_ctas must be 0; MXFP8 and
                                   split_k >= 2 return BST_ERR_UNSUPPORTED.          */
} bst_sched;

/*
 * bst_gemm -- C[M,N] = A[M,K] . B[K,N] ("Block Dispatch Policies",
 * 00_basic_matmul), accumulated in fp32, rounded once to the type of C.
 *
 *   a_type == b_type == BST_F16 or BST_BF16: c_type BST_F16, BST_BF16 or
 *     BST_F32; any layout for A and B; scale_a/scale_b must be NULL.
 *   a_type == b_type == BST_E4M3 (MXFP8): A row-major, B column-major (both
 *     K-contiguous), K a multiple of 128, c_type BST_BF16, BST_F16 or
 *     BST_F32; scale_a [M, K/32] and scale_b [N, K/32] are dense row-major
 *     E8M0 codes (value 2^(s-127)), one per 32 consecutive K elements of a
 *     row of A / a column of B.
 * ldc >= N.  C must not overlap A or B.
 * Returns BST_OK once the launch is enqueued.
 */
bst_status bst_gemm(int64_t M, int64_t N, int64_t K,
                    const void* A, bst_dtype a_type, bst_layout a_layout, int64_t lda,
                    const void* B, bst_dtype b_type, bst_layout b_layout, int64_t ldb,
                    void* C, bst_dtype c_type, int64_t ldc,
                    const uint8_t* scale_a, const uint8_t* scale_b,
                    const bst_sched* sched, void* stream);

/*
 * bst_gemm_batched -- `batch` independent bst_gemm problems of one shape
 * ("Block Dispatch Policies", 01_batched_matmul; task t belongs to batch
 * t / (loopsM*loopsN), "Block Scheduler Code Explained" section 4.4
 * GetBatchIdx).  Problem i uses A + i*stride_a, B + i*stride_b,
 * C + i*stride_c (strides in elements; for TMA they must be 16-byte
 * multiples).  fp16/bf16 operands only.
 */
bst_status bst_gemm_batched(int64_t M, int64_t N, int64_t K,
                            const void* A, bst_dtype a_type, bst_layout a_layout, int64_t lda, int64_t stride_a,
                            const void* B, bst_dtype b_type, bst_layout b_layout, int64_t ldb, int64_t stride_b,
                            void* C, bst_dtype c_type, int64_t ldc, int64_t stride_c,
                            int64_t batch, const bst_sched* sched, void* stream);

/*
 * bst_gemm_grouped -- grouped GEMM with groups along M ("Block Dispatch
 * Policies", 02_grouped_matmul_slice_m).  Group g owns the M_g consecutive
 * rows [off_g, off_g + M_g) of A and of C, off_g = M_0 + ... + M_{g-1}, and
 * multiplies them by its own B_g:
 *
 *   C[off_g + i, :] = A[off_g + i, :] . B_g      for 0 <= i < M_g.
 *
 * group_m  DEVICE int32[G] of group sizes (>= 0; zero-size groups own no
 *          rows).  The host never reads it, so no synchronisation is implied.
 * total_m  rows of the A and C buffers; the kernel checks sum(M_g) <= total_m
 *          and otherwise computes nothing and records BST_ERR_DEVICE.
 * A        [total_m, K] row-major (lda).
 * B        G matrices; b_layout BST_ROW_MAJOR: B_g is [K, N] at
 *          B + g*stride_b with leading dimension ldb (N contiguous);
 *          BST_COL_MAJOR: stored [N, K] (K contiguous).
 * C        [total_m, N] row-major (ldc); rows past sum(M_g) are not written.
 * dtype    BST_F16 or BST_BF16 for A and B; c_type BST_F16, BST_BF16, BST_F32.
 * Tasks are numbered group-major and the swizzle restarts in each group, as
 * "Block Scheduler Code Explained" section 4.2 (Update) re-targets the
 * scheduler to (M_g, N, K).  G <= 1024.
 */
bst_status bst_gemm_grouped(int32_t G, const int32_t* group_m, int64_t total_m,
                            int64_t N, int64_t K,
                            const void* A, int64_t lda,
                            const void* B, bst_layout b_layout, int64_t ldb, int64_t stride_b,
                            void* C, int64_t ldc,
                            bst_dtype ab_type, bst_dtype c_type,
                            const bst_sched* sched, void* stream);

/*
 * bst_gemm_quant_per_token -- int8 GEMM with per-token dequant ("Block
 * Dispatch Policies", 12_quant_matmul):
 *
 *   acc[i,j] = sum_k A[i,k] * B[k,j]          exactly, in int32
 *   C[i,j]   = bf16( acc[i,j] * scale_a[i] * scale_b[j] )    (fp32 products)
 *
 * A int8 [M, K] row-major (lda); B int8 with b_layout (BST_COL_MAJOR: stored
 * [N, K], the usual weight layout).  scale_a fp32 [M] (one per row/token),
 * scale_b fp32 [N] (one per output column).  C bf16 [M, N] (ldc).
 * acc_out: optional int32 [M, N] row-major with leading dimension ldc that
 * receives the exact accumulators (NULL = not written).
 * workspace: DEVICE scratch of at least
 * bst_gemm_quant_per_token_workspace_size(M, N, K) bytes, 256-byte aligned,
 * owned by the caller and not read after the call's kernels finish; calls
 * that share one workspace must be ordered on one stream.  The operands are
 * widened to bf16 there (every int8 is exact in bf16) and multiplied on the
 * tensor cores in K-chunks of at most 1024, each chunk's fp32 sum being an
 * exact integer below 2^24, carried into int32.
 */
size_t bst_gemm_quant_per_token_workspace_size(int64_t M, int64_t N, int64_t K);

bst_status bst_gemm_quant_per_token(int64_t M, int64_t N, int64_t K,
                                    const int8_t* A, int64_t lda,
                                    const int8_t* B, bst_layout b_layout, int64_t ldb,
                                    const float* scale_a, const float* scale_b,
                                    void* C, int64_t ldc, int32_t* acc_out,
                                    void* workspace, size_t workspace_bytes,
                                    const bst_sched* sched, void* stream);

/*
 * bst_gemm_grouped_quant_per_token -- grouped slice-M int8 GEMM with
 * per-token dequant ("Block Dispatch Policies",
 * 10_grouped_matmul_slice_m_per_token_dequant): for every group g, rows
 * [off_g, off_g + M_g) of A and C (off_g = the sum of the earlier sizes) use
 * B_g and the column scales of group g:
 *
 *   acc[i,j] = sum_k A[i,k] * B_g[k,j]         exactly, in int32
 *   C[i,j]   = bf16( acc[i,j] * scale_a[i] * scale_b[g*stride_sb + j] )
 *
 * group_m: DEVICE int32 [G] (zero-size groups allowed; 1 <= G <= 1024), whose
 * sum must equal total_m (else bst_check_async reports BST_ERR_DEVICE and no
 * tile is computed).  A int8 [total_m, K] row-major (lda).  B: G matrices
 * int8, stride_b elements apart, each [N, K] (BST_COL_MAJOR) or [K, N]
 * (BST_ROW_MAJOR) with leading dimension ldb.  scale_a fp32 [total_m];
 * scale_b fp32 [G, N] with row stride stride_sb.  C bf16 [total_m, N] (ldc);
 * acc_out optional int32 [total_m, N] with ldc.  workspace: DEVICE scratch of
 * bst_gemm_grouped_quant_per_token_workspace_size(G, total_m, N, K) bytes,
 * 256-byte aligned, caller-owned; the operands are widened to bf16 there and
 * multiplied exactly on 256 x 256 CTA-pair tiles (as bst_gemm_quant_per_token
 * does), tasks numbered group-major with the swizzle restarted per group.
 */
size_t bst_gemm_grouped_quant_per_token_workspace_size(int32_t G, int64_t total_m, int64_t N, int64_t K);

bst_status bst_gemm_grouped_quant_per_token(int32_t G, const int32_t* group_m, int64_t total_m, int64_t N, int64_t K,
                                            const int8_t* A, int64_t lda,
                                            const int8_t* B, bst_layout b_layout, int64_t ldb, int64_t stride_b,
                                            const float* scale_a, const float* scale_b, int64_t stride_sb,
                                            void* C, int64_t ldc, int32_t* acc_out,
                                            void* workspace, size_t workspace_bytes,
                                            const bst_sched* sched, void* stream);

/*
 * bst_gemm_grouped_slice_k -- grouped GEMM with groups along K ("Block
 * Dispatch Policies", 05_grouped_matmul_slice_k).  Group g owns the K_g
 * consecutive K indices [off_g, off_g + K_g) of A and B, off_g = K_0 + ... +
 * K_{g-1}, and produces its own output matrix:
 *
 *   C_g = A[:, off_g : off_g + K_g] . B[off_g : off_g + K_g, :]      ([M, N])
 *
 * (e.g. a weight gradient X_g^T . dY_g whose groups are runs of tokens).
 * group_k  DEVICE int32[G], 1 <= G <= 1024.  Zero-size groups give C_g = 0.
 *          The kernel checks the sizes (none negative, sum <= total_k, and,
 *          where an operand is K-contiguous, every non-empty group starting
 *          on a 16-byte boundary: off_g a multiple of 8); otherwise nothing is
 *          written and bst_check_async reports BST_ERR_DEVICE.  K indices past
 *          the sum are not read.
 * A        logical [M, total_k]; a_layout BST_ROW_MAJOR: stored [M, total_k]
 *          (K contiguous); BST_COL_MAJOR: stored [total_k, M] (M contiguous,
 *          the layout of X in X^T . dY).  Leading dimension lda.
 * B        logical [total_k, N]; BST_ROW_MAJOR: stored [total_k, N] (N
 *          contiguous); BST_COL_MAJOR: stored [N, total_k].  Leading dim ldb.
 * C        G row-major [M, N] matrices (ldc), C_g at C + g*stride_c elements
 *          (stride_c >= M*ldc when G > 1).
 * dtype    ab_type BST_F16 or BST_BF16; c_type BST_F16, BST_BF16 or BST_F32.
 * workspace DEVICE scratch of bst_gemm_grouped_slice_k_workspace_size(G)
 *          bytes, 256-byte aligned, caller-owned: per group a copy of each
 *          operand's TMA map rewritten on the device (base at off_g, K extent
 *          K_g, so a group's ragged last k-block reads zeros), and the
 *          groups' k-block counts.
 * Runs on 256 x 256 or 256 x 128 CTA-pair tiles; tasks are numbered
 * group-major (task t belongs to group t / (loopsM*loopsN), as batches are in
 * "Block Scheduler Code Explained" section 4.4) with the swizzle of every
 * group over the same M x N grid.  Operands must be TMA-addressable (16-byte
 * aligned base and leading dimension), else BST_ERR_ALIGNMENT.  total_k = 0:
 * every C_g is zeroed.
 */
size_t bst_gemm_grouped_slice_k_workspace_size(int32_t G);

bst_status bst_gemm_grouped_slice_k(int32_t G, const int32_t* group_k, int64_t M, int64_t N, int64_t total_k,
                                    const void* A, bst_layout a_layout, int64_t lda,
                                    const void* B, bst_layout b_layout, int64_t ldb,
                                    void* C, int64_t ldc, int64_t stride_c,
                                    bst_dtype ab_type, bst_dtype c_type,
                                    void* workspace, size_t workspace_bytes,
                                    const bst_sched* sched, void* stream);

/*
 * bst_gemm_grouped_slice_k_quant_per_token -- the K slices of
 * bst_gemm_grouped_slice_k on int8 operands, each group dequantised with its
 * own scales ("Block Dispatch Policies",
 * 11_grouped_matmul_slice_k_per_token_dequant):
 *
 *   acc_g[i,j] = sum over k in slice g of A[i,k] * B[k,j]     exactly, int32
 *   C_g[i,j]   = bf16( acc_g[i,j] * scale_a[g*stride_sa + i] * scale_b[g*stride_sb + j] )
 *
 * scale_a fp32 [G, M] (row stride stride_sa; 0 shares one row of scales),
 * scale_b fp32 [G, N] (stride_sb).  A, B, group_k and the layouts as for
 * bst_gemm_grouped_slice_k (int8 elements).  C bf16, acc_out optional int32,
 * both G x [M, N] with ldc and stride_c.  workspace: DEVICE scratch of
 * bst_gemm_grouped_slice_k_quant_per_token_workspace_size(G, M, N, total_k)
 * bytes, 256-byte aligned: the per-group maps plus A and B widened to bf16,
 * multiplied exactly as bst_gemm_quant_per_token does on 256 x 256 pairs.
 */
size_t bst_gemm_grouped_slice_k_quant_per_token_workspace_size(int32_t G, int64_t M, int64_t N, int64_t total_k);

bst_status bst_gemm_grouped_slice_k_quant_per_token(int32_t G, const int32_t* group_k, int64_t M, int64_t N,
                                                    int64_t total_k,
                                                    const int8_t* A, bst_layout a_layout, int64_t lda,
                                                    const int8_t* B, bst_layout b_layout, int64_t ldb,
                                                    const float* scale_a, int64_t stride_sa,
                                                    const float* scale_b, int64_t stride_sb,
                                                    void* C, int64_t ldc, int64_t stride_c, int32_t* acc_out,
                                                    void* workspace, size_t workspace_bytes,
                                                    const bst_sched* sched, void* stream);

/*
 * bst_gemm_quant_per_token_noalloc -- the same int8 GEMM with per-token
 * dequant as bst_gemm_quant_per_token (same arguments, results and errors),
 * for callers that cannot allocate device memory at the point of the call:
 * a plain C host program that has no device allocator of its own, or a
 * process whose device memory is already reserved by another framework's
 * pool, where an extra allocation would fail or fragment that pool.  The
 * pages have no counterpart of this entry point; it exists for such callers.
 *
 * Instead of a caller-owned workspace it uses one scratch array of
 * BST_NOALLOC_SCRATCH_BYTES compiled into the library, and it allocates
 * nothing (no cudaMalloc, no library allocator).  A problem whose
 * bst_gemm_quant_per_token_workspace_size(M, N, K) exceeds that limit is
 * rejected with BST_ERR_UNSUPPORTED before any CUDA call.  The first call on
 * each device looks up the array's device address with that device current
 * (a one-time set-up, not repeated); make that first call before any stream
 * capture.  Every call on a device shares the one array: calls on the same
 * stream run one after another and are safe, while calls that can overlap
 * (different streams, or host threads without ordering between their
 * streams) race on the scratch and give wrong results.
 */
#define BST_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

bst_status bst_gemm_quant_per_token_noalloc(int64_t M, int64_t N, int64_t K,
                                            const int8_t* A, int64_t lda,
                                            const int8_t* B, bst_layout b_layout, int64_t ldb,
                                            const float* scale_a, const float* scale_b,
                                            void* C, int64_t ldc, int32_t* acc_out,
                                            const bst_sched* sched, void* stream);

/*
 * bst_swizzle_map -- debug entry: runs the device scheduler the GEMM kernels
 * use ("Block Scheduler Code Explained" sections 4.3-4.6) for every task of a
 * (possibly batched) problem and writes, for task t, the 5 uint32
 * {GetBatchIdx, mIdx, nIdx, mActual, nActual} to out[5*t .. 5*t+4].
 * out is a DEVICE buffer of 5 * batch * ceil(M/tile_m) * ceil(N/tile_n)
 * uint32.  Any tile sizes >= 1 are accepted.  The task count must be < 2^32.
 */
bst_status bst_swizzle_map(uint32_t M, uint32_t N, uint32_t tile_m, uint32_t tile_n,
                           uint32_t batch, const bst_sched* sched,
                           uint32_t* out, void* stream);

/*
 * bst_swizzle_map_grouped -- the same for a grouped slice-M problem: group
 * sizes are read from DEVICE int32 group_m[G]; task t (group-major) gets
 * {group, mIdx, nIdx, mActual, nActual}.  out holds max_tasks rows; tasks
 * past max_tasks are not written (bst_check_async then reports
 * BST_ERR_DEVICE).
 */
bst_status bst_swizzle_map_grouped(int32_t G, const int32_t* group_m, uint32_t N,
                                   uint32_t tile_m, uint32_t tile_n, const bst_sched* sched,
                                   uint32_t* out, uint32_t max_tasks, void* stream);

/*
 * bst_check_async -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns BST_ERR_TIMEOUT if a kernel's bounded
 * wait gave up, BST_ERR_DEVICE if a device-side check failed, BST_ERR_CUDA
 * if the stream reported an error, else BST_OK.
 */
bst_status bst_check_async(void* stream);

/* A short static English description of a status code. */
const char* bst_status_string(bst_status s);

/*
 * bst_set_wait_timeout_ns -- limit, in nanoseconds, on every device-side
 * wait of kernels launched afterwards by this thread (0 = the default of
 * 4 s).  Used by tests to make a wait that cannot complete give up quickly.
 */
void bst_set_wait_timeout_ns(uint64_t ns);

/*
 * bst_wait_check -- self-check of the device-side failure detection (the
 * pages have no counterpart; it exercises the bounded waits every GEMM kernel
 * uses between its producer, MMA and epilogue roles).  Launches one small
 * kernel on `stream` whose thread waits on a shared-memory barrier with that
 * bounded wait.  arrive != 0: another thread arrives on the barrier first, so
 * the wait succeeds and the next bst_check_async returns BST_OK.  arrive == 0:
 * nothing arrives, the wait gives up after timeout_ns (1 ns .. 10 s, else
 * BST_ERR_INVALID_ARG before anything is launched) and the next
 * bst_check_async returns BST_ERR_TIMEOUT.  Nothing else is in flight while
 * it waits, so the device stays usable.  Asynchronous; allocates nothing.
 */
bst_status bst_wait_check(uint64_t timeout_ns, int32_t arrive, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BST_H */
