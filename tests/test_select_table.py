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
