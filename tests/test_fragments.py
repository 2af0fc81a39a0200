"""The m16n8k16 fragment formulas (tests/fragments.py) against the tables the
page prints, and the covering property every fragment layout must have
(CPU only; the GPU test checks them against the hardware)."""
import json
import os

import fragments as fr

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "m16n8k16_fragments.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_formulas_reproduce_printed_a_rows():
    for lane, g, t, ranges in _golden()["A"]:
        assert (lane >> 2, lane % 4) == (g, t)
        for pair, (row, c0, c1) in enumerate(ranges):
            assert fr.a_coord(lane, 2 * pair) == (row, c0)
            assert fr.a_coord(lane, 2 * pair + 1) == (row, c1)


def test_formulas_reproduce_printed_b_rows():
    for lane, g, t, ranges in _golden()["B"]:
        assert (lane >> 2, lane % 4) == (g, t)
        for pair, (r0, r1, col) in enumerate(ranges):
            assert fr.b_coord(lane, 2 * pair) == (r0, col)
            assert fr.b_coord(lane, 2 * pair + 1) == (r1, col)


def test_formulas_reproduce_printed_c_rows():
    for lane, g, t, ranges in _golden()["C"]:
        assert (lane >> 2, lane % 4) == (g, t)
        for pair, (row, c0, c1) in enumerate(ranges):
            assert fr.c_coord(lane, 2 * pair) == (row, c0)
            assert fr.c_coord(lane, 2 * pair + 1) == (row, c1)


def test_each_element_held_exactly_once():
    """A 16 x 16 = 32 lanes x 8, B 16 x 8 = 32 x 4, C 16 x 8 = 32 x 4."""
    for coord, n_el, rows, cols in ((fr.a_coord, 8, 16, 16), (fr.b_coord, 4, 16, 8), (fr.c_coord, 4, 16, 8)):
        seen = sorted(coord(l, i) for l in range(32) for i in range(n_el))
        assert seen == [(r, c) for r in range(rows) for c in range(cols)]
