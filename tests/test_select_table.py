"""The kernel-path selection table (no GPU): the rule that turns a measured
sweep into per-shape limits, and the committed header's agreement with the
committed sweep it was generated from."""
import os

import pytest

from quantized_allreduce_codec_gb300 import select_table as st


def test_limit_is_the_crossover_of_a_clean_sweep():
    # direct faster up to 1M elements, pipeline faster beyond
    pts = [(n, 1.0 if n <= 1 << 20 else 3.0, 2.0) for n in (1 << k for k in range(10, 26))]
    assert st.choose_limit(pts) == 1 << 20


def test_all_pipeline_and_all_direct():
    sizes = [1 << k for k in range(10, 26)]
    assert st.choose_limit([(n, 2.0, 1.0) for n in sizes]) == 0
    # the direct kernel wins at the largest size measured: every size
    assert st.choose_limit([(n, 1.0, 2.0) for n in sizes]) == st.MAX_ELEMS


def test_one_noisy_point_does_not_move_the_limit():
    sizes = [1 << k for k in range(10, 26)]
    pts = []
    for n in sizes:
        td, tp = (1.0, 2.0) if n <= 1 << 18 else (2.0, 1.0)
        if n == 1 << 22:
            td, tp = 0.99, 1.0  # a lone point where the direct kernel edges ahead
        pts.append((n, td, tp))
    assert st.choose_limit(pts) == 1 << 18


def test_ties_go_to_the_smaller_limit():
    assert st.choose_limit([(1024, 1.0, 1.0), (2048, 1.0, 1.0)]) == 0


def test_three_way_limits_are_the_two_crossovers_of_a_clean_sweep():
    # direct fastest up to 1M elements, narrow tiles up to 16M, wide tiles beyond
    def t(n):
        return (1.0 if n <= 1 << 20 else 3.0, 2.0 if n <= 1 << 24 else 4.0, 2.5 if n <= 1 << 24 else 1.0)
    pts = [(n, *t(n)) for n in (1 << k for k in range(10, 27))]
    assert st.choose_limits(pts) == (1 << 20, 1 << 24)


def test_narrow_tiles_that_never_win_get_an_empty_range():
    pts = [(n, 1.0 if n <= 1 << 20 else 3.0, 2.5, 2.0) for n in (1 << k for k in range(10, 26))]
    l1, l2 = st.choose_limits(pts)
    assert l1 == 1 << 20 and l2 == l1


def test_narrow_tiles_winning_at_the_largest_size_extend_to_every_size():
    pts = [(n, 1.0 if n <= 1 << 20 else 3.0, 2.0, 2.5) for n in (1 << k for k in range(10, 26))]
    assert st.choose_limits(pts) == (1 << 20, st.MAX_ELEMS)


def test_without_narrow_timings_the_limits_coincide():
    pts = [(n, 1.0 if n <= 1 << 18 else 2.0, None, 1.5) for n in (1 << k for k in range(10, 26))]
    assert st.choose_limits(pts) == (1 << 18, 1 << 18)


def test_tables_carry_both_limits():
    lim = {(0, 2, 2, 3): (1 << 20, 1 << 24)}
    assert st.table(lim, 0)[0][2][1][3] == 1 << 20
    assert st.table(lim, 1)[0][2][1][3] == 1 << 24
    text = st.render(st.table(lim, 0), st.table(lim, 1), "x.json")
    assert "kDirectLimitTable[3][3][4][7]" in text and "kNarrowTileLimitTable[3][3][4][7]" in text


def test_table_shape_and_impossible_shapes():
    tab = st.table({})
    assert len(tab) == 3 and all(len(a) == 3 for a in tab)
    assert all(len(b) == 4 and all(len(r) == 7 for r in b) for a in tab for b in a)
    assert tab[2][0] == [[0] * 7] * 4            # the cast option has no encode-only call
    assert tab[0][0][1] == [0] * 7               # encode-only runs one rank
    assert tab[0][2][3][3] == st.DEFAULT_LIMIT   # a shape the sweep did not cover


@pytest.mark.skipif(not os.path.exists(st.SWEEP), reason="no committed sweep yet")
def test_committed_header_is_generated_from_the_committed_sweep():
    assert open(st.HEADER).read() == st.generate(st.SWEEP)
