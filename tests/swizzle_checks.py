"""Properties any correct task -> tile map of GemmIdentityBlockSwizzle has
("Block Scheduler Code Explained", sections 4.5, 4.6 and 5), written as
checkers that return a list of violations.  Used to pin the oracle and, on the
GPU, to check the device scheduler's output independently of the oracle."""
import os

from oracle.swizzle import ceil_div

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "swizzle_examples.txt")


def load_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case"):
                _, name, *nums = line.split()
                M, N, tm, tn, S, d = map(int, nums)
                cur = dict(name=name, M=M, N=N, tile_m=tm, tile_n=tn, offset=S, direction=d, rows=[])
                cases.append(cur)
            else:
                cur["rows"].append(tuple(map(int, line.split())))
    return cases


def check_map(rows, M, N, tile_m, tile_n, offset, direction):
    """rows: list of (m, n, mActual, nActual) for tasks 0..coreLoops-1."""
    v = []
    lm, ln = ceil_div(M, tile_m), ceil_div(N, tile_n)
    if len(rows) != lm * ln:
        return ["expected %d tasks, got %d" % (lm * ln, len(rows))]
    # bijection onto the tile grid
    seen = set((r[0], r[1]) for r in rows)
    if len(seen) != lm * ln or any(not (0 <= m < lm and 0 <= n < ln) for m, n in seen):
        v.append("not a bijection onto the %dx%d grid" % (lm, ln))
    # exact cover of M x N by the actual shapes
    area = 0
    for m, n, ma, na in rows:
        if not (0 < ma <= tile_m and 0 < na <= tile_n):
            v.append("bad actual shape %s" % ((m, n, ma, na),))
        if m * tile_m + ma > M or n * tile_n + na > N:
            v.append("tile %s leaves the problem" % ((m, n, ma, na),))
        if m < lm - 1 and ma != tile_m or n < ln - 1 and na != tile_n:
            v.append("interior tile cut %s" % ((m, n, ma, na),))
        area += ma * na
    if area != M * N:
        v.append("tiles cover %d elements, problem has %d" % (area, M * N))
    # window structure and snake
    S = offset
    if direction == 0:
        outer, inner = lm, ln
        key = lambda r: (r[0], r[1])          # (window axis, sweep axis)
    else:
        outer, inner = ln, lm
        key = lambda r: (r[1], r[0])
    W = ceil_div(outer, S)
    t = 0
    for w in range(W):
        h = min(S, outer - w * S)
        chunk = [key(r) for r in rows[t:t + h * inner]]
        t += h * inner
        want = set((w * S + i, j) for i in range(h) for j in range(inner))
        if set(chunk) != want:
            v.append("window %d does not hold exactly lines %d..%d" % (w, w * S, w * S + h - 1))
            continue
        # inside a window the window axis runs fastest, the sweep axis in order
        sweep = list(range(inner)) if w % 2 == 0 else list(range(inner - 1, -1, -1))
        expect = [(w * S + i, j) for j in sweep for i in range(h)]
        if chunk != expect:
            v.append("window %d order/snake wrong" % w)
    return v


def closed_form(t, lm, ln, offset, direction):
    """Orders the page's definition reduces to in its limiting cases."""
    if direction == 0 and offset >= lm:
        return t % lm, t // lm                 # one window: column-major
    if direction == 0 and offset == 1:
        m, j = t // ln, t % ln                 # one tile-row per window: boustrophedon
        return m, (j if m % 2 == 0 else ln - 1 - j)
    if direction == 1 and offset >= ln:
        return t // ln, t % ln                 # one window: row-major
    if direction == 1 and offset == 1:
        n, i = t // lm, t % lm
        return (i if n % 2 == 0 else lm - 1 - i), n
    return None
