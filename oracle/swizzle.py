"""Task index -> output tile, as GemmIdentityBlockSwizzle defines it.
TEST INFRASTRUCTURE ONLY.

Source: "Block Scheduler Code Explained" (CATLASS docs), section 2.1 (template
parameters SwizzleOffset, default 1, and SwizzleDirection, 0 = Zn, 1 = Nz),
section 3 (state: problem shape, tile shape, loop counts), section 4.1
(loop counts are the ceiling division of the problem's M, N by the tile's),
section 4.2 (Update re-targets the shape), 4.3 GetCoreLoops, 4.4 GetBatchIdx,
4.5 GetBlockCoord, 4.6 GetActualBlockShape, section 5 (window-based
scheduling, snake scanning, tail blocks) and section 6
(DynamicGemmIdentityBlockSwizzle: offset and direction chosen at run time).

All arithmetic is on exact Python integers, so no wrap-around of the page's
uint32 products can occur here.

Readings taken where the page is silent:
* CeilDiv is never printed: it is the integer ceiling ceil(a / b).
* The Nz body of GetBlockCoord is elided: the page only says it mirrors the
  Zn logic.  Section 4.5's prose gives Nz windows a width of SwizzleOffset
  tile-columns and has the snake reverse the index of whichever dimension the
  window runs along; the reading taken is the exact transpose of the Zn
  branch: windows of SwizzleOffset tile-columns, n fastest inside a window,
  the last window narrower, m reversed on odd windows.  Parity of this branch is pinned only
  by invariants and closed forms (bijection, exact cover, window shape,
  snake, row-major order when SwizzleOffset >= loopsN).
* GemmCoord{mIdx, nIdx, 0} are tile indices; the tile's first element is
  (mIdx * tileM, nIdx * tileN).
* Grouped slice-M ("Block Dispatch Policies", MmadAtlasA2PreloadAsync,
  example 02_grouped_matmul_slice_m, plus Update in section 4.2): tasks are
  numbered group-major, and the scheduler is re-targeted with Update to
  (M_g, N, K) for each group, so the swizzle restarts inside each group.
  Groups with M_g == 0 own no task.
"""


def ceil_div(a, b):
    """Integer ceiling of a / b (the page's CeilDiv, section 4.1)."""
    return (a + b - 1) // b


class IdentityBlockSwizzle:
    """State and methods of GemmIdentityBlockSwizzle (sections 3 and 4),
    with the run-time offset/direction of the dynamic variant (section 6)."""

    def __init__(self, M, N, K, tile_m, tile_n, swizzle_offset=1, swizzle_direction=0):
        if swizzle_offset < 1:
            raise ValueError("SwizzleOffset must be >= 1")
        if swizzle_direction not in (0, 1):
            raise ValueError("SwizzleDirection must be 0 (Zn) or 1 (Nz)")
        self.swizzle_offset = swizzle_offset
        self.swizzle_direction = swizzle_direction
        self.update(M, N, K, tile_m, tile_n)

    def update(self, M, N, K, tile_m, tile_n):
        """Section 4.2: new problem and tile shape, loop counts recomputed."""
        self.M, self.N, self.K = M, N, K
        self.tile_m, self.tile_n = tile_m, tile_n
        self.loops_m = ceil_div(M, tile_m)
        self.loops_n = ceil_div(N, tile_n)

    def core_loops(self):
        """Section 4.3: tiles per batch = loopsM * loopsN."""
        return self.loops_m * self.loops_n

    def batch_idx(self, task):
        """Section 4.4: which batch a task index belongs to."""
        return task // self.core_loops()

    def block_coord(self, task):
        """Section 4.5: (mIdx, nIdx) of the tile that ``task`` computes."""
        inner = task % self.core_loops()
        S = self.swizzle_offset
        if self.swizzle_direction == 0:                      # Zn
            n_windows = ceil_div(self.loops_m, S)
            window = inner // (S * self.loops_n)
            pos = inner % (S * self.loops_n)
            rows = S
            if window == n_windows - 1:                      # short last window
                rows = self.loops_m - S * window
            m = window * S + pos % rows                      # m runs fastest
            n = pos // rows
            if window % 2 == 1:                              # snake
                n = self.loops_n - n - 1
            return m, n
        # Nz: the transpose of the Zn branch (reading stated in the module doc)
        n_windows = ceil_div(self.loops_n, S)
        window = inner // (S * self.loops_m)
        pos = inner % (S * self.loops_m)
        cols = S
        if window == n_windows - 1:
            cols = self.loops_n - S * window
        n = window * S + pos % cols                          # n runs fastest
        m = pos // cols
        if window % 2 == 1:
            m = self.loops_m - m - 1
        return m, n

    def actual_block_shape(self, m, n):
        """Section 4.6: the tile's real extent; the last tile-row/column is cut
        to what is left of the problem.  kActual is the whole K."""
        m_act = self.M - m * self.tile_m if m == self.loops_m - 1 else self.tile_m
        n_act = self.N - n * self.tile_n if n == self.loops_n - 1 else self.tile_n
        return m_act, n_act, self.K


def swizzle_map(M, N, tile_m, tile_n, swizzle_offset=1, swizzle_direction=0, batch=1, K=0):
    """Rows (batch, m, n, mActual, nActual) for task 0 .. batch*coreLoops-1,
    following the execution flow of section 7: batch index, block coordinate,
    actual block shape, per task."""
    sch = IdentityBlockSwizzle(M, N, K, tile_m, tile_n, swizzle_offset, swizzle_direction)
    rows = []
    for t in range(batch * sch.core_loops()):
        b = sch.batch_idx(t)
        m, n = sch.block_coord(t)
        ma, na, _ = sch.actual_block_shape(m, n)
        rows.append((b, m, n, ma, na))
    return rows


def grouped_swizzle_map(group_m, N, tile_m, tile_n, swizzle_offset=1, swizzle_direction=0, K=0):
    """Rows (group, m, n, mActual, nActual) for every task of a grouped
    slice-M problem: groups in order, the scheduler re-targeted per group
    (section 4.2 Update) to (M_g, N, K)."""
    rows = []
    sch = IdentityBlockSwizzle(1, N, K, tile_m, tile_n, swizzle_offset, swizzle_direction)
    for g, mg in enumerate(group_m):
        if mg == 0:
            continue
        sch.update(mg, N, K, tile_m, tile_n)
        for t in range(sch.core_loops()):
            m, n = sch.block_coord(t)
            ma, na, _ = sch.actual_block_shape(m, n)
            rows.append((g, m, n, ma, na))
    return rows
