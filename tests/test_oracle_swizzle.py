"""Pins for oracle.swizzle (GemmIdentityBlockSwizzle, "Block Scheduler Code
Explained" sections 4-6): hand-derived worked examples, invariants (bijection,
exact cover, windows, snake), closed forms, and planted mistakes that the
invariants must catch."""
import itertools

import pytest

from oracle import swizzle as osw
from tests.swizzle_checks import check_map, closed_form, load_golden

SHAPES = [(500, 380, 128, 128), (1024, 1024, 128, 128), (1024, 1024, 128, 256),
          (8192, 8192, 128, 256), (1, 1, 128, 128), (129, 2000, 128, 64),
          (48, 74, 16, 16), (80, 48, 16, 16), (1000, 37, 16, 8), (7, 700, 8, 16)]
OFFSETS = [1, 2, 3, 4, 5, 8, 9, 1000]


def _rows(M, N, tm, tn, S, d):
    return [r[1:] for r in osw.swizzle_map(M, N, tm, tn, S, d)]


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_worked_examples(case):
    got = _rows(case["M"], case["N"], case["tile_m"], case["tile_n"], case["offset"], case["direction"])
    assert got == case["rows"]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("S", OFFSETS)
@pytest.mark.parametrize("d", [0, 1])
def test_invariants(shape, S, d):
    M, N, tm, tn = shape
    assert check_map(_rows(M, N, tm, tn, S, d), M, N, tm, tn, S, d) == []


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("d", [0, 1])
def test_closed_forms(shape, d):
    M, N, tm, tn = shape
    lm, ln = osw.ceil_div(M, tm), osw.ceil_div(N, tn)
    for S in (1, lm if d == 0 else ln, 10 ** 6):
        rows = _rows(M, N, tm, tn, S, d)
        for t, r in enumerate(rows):
            cf = closed_form(t, lm, ln, S, d)
            assert cf is not None and r[:2] == cf, (S, t, r, cf)


def test_offset_beyond_loops_equals_offset_loops():
    # once SwizzleOffset >= loopsM (Zn) there is a single window; larger values
    # give the same map
    for (M, N, tm, tn), d in itertools.product(SHAPES, [0, 1]):
        lm, ln = osw.ceil_div(M, tm), osw.ceil_div(N, tn)
        lim = lm if d == 0 else ln
        assert _rows(M, N, tm, tn, lim, d) == _rows(M, N, tm, tn, lim + 7, d)


def test_batch_index_and_repeat():
    rows = osw.swizzle_map(500, 380, 128, 128, 3, 0, batch=3)
    core = 12
    assert [r[0] for r in rows] == [t // core for t in range(36)]
    for t in range(36):
        assert rows[t][1:] == rows[t % core][1:]


def test_grouped_is_concatenation_of_updated_maps():
    gm = [0, 300, 0, 129, 1, 0, 1024]
    rows = osw.grouped_swizzle_map(gm, 700, 128, 128, 2, 0)
    want = []
    for g, mg in enumerate(gm):
        if mg:
            want += [(g,) + r[1:] for r in osw.swizzle_map(mg, 700, 128, 128, 2, 0)]
    assert rows == want
    assert {r[0] for r in rows} == {1, 3, 4, 6}


def test_rejects_bad_params():
    with pytest.raises(ValueError):
        osw.IdentityBlockSwizzle(10, 10, 1, 4, 4, 0, 0)
    with pytest.raises(ValueError):
        osw.IdentityBlockSwizzle(10, 10, 1, 4, 4, 1, 2)


# ---- planted mistakes: each must be caught by the checks used above -------

def _mutant(kind):
    class Mut(osw.IdentityBlockSwizzle):
        def block_coord(self, task):
            inner = task % self.core_loops()
            S, lm, ln = self.swizzle_offset, self.loops_m, self.loops_n
            W = osw.ceil_div(lm, S)
            w = inner // (S * ln)
            pos = inner % (S * ln)
            rows = S if (w != W - 1 or kind == "full_last_window") else lm - S * w
            m = w * S + pos % rows
            n = pos // rows
            if kind == "n_fastest":
                m, n = w * S + pos // ln, pos % ln
            if w % 2 == 1 and kind != "no_snake":
                n = ln - n - 1
            if kind == "snake_on_even" and w % 2 == 0:
                n = ln - n - 1
            return m, n

        def actual_block_shape(self, m, n):
            ma, na, k = super().actual_block_shape(m, n)
            if kind == "tail_off_by_one" and m == self.loops_m - 1:
                ma += 1
            return ma, na, k
    return Mut


@pytest.mark.parametrize("kind", ["no_snake", "full_last_window", "n_fastest",
                                  "snake_on_even", "tail_off_by_one"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(osw, "IdentityBlockSwizzle", _mutant(kind))
    caught = False
    for (M, N, tm, tn), S in itertools.product(SHAPES, [2, 3]):
        rows = [r[1:] for r in osw.swizzle_map(M, N, tm, tn, S, 0)]
        if check_map(rows, M, N, tm, tn, S, 0):
            caught = True
            break
    gold = [c for c in load_golden() if c["direction"] == 0]
    caught_gold = any(
        [r[1:] for r in osw.swizzle_map(c["M"], c["N"], c["tile_m"], c["tile_n"], c["offset"], 0)] != c["rows"]
        for c in gold)
    assert caught and caught_gold
