"""The bench's host-side reports, without a GPU: the deviation-from-exact-sum
report accepts the oracle's own outputs (which meet the stated bounds by the
oracle pins) and rejects an output with a planted error, and the per-recipe
oracle timing covers every workload, format and stage count."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantized_allreduce_codec_gb300.inputs import (BF16, F16, FP, Q4, Workload,  # noqa: E402
                                                    sweep_workload, to_bits, workloads)


@pytest.mark.parametrize("size_bytes", [1 << 16, 1 << 20])
def test_oracle_outputs_meet_the_reported_bounds(oracle_mod, size_bytes):
    wl = sweep_workload(size_bytes)
    host = wl.inputs()
    for fmt, st in bench.TP2_CALLS:
        out, _ = oracle_mod.allreduce(wl.dtype, fmt, st, host)
        rep = bench.error_vs_exact(host, out, wl.dtype, fmt, st)
        assert rep["within_bound_fraction"] == 1.0, (fmt, st, rep)
        assert rep["max_abs"] >= 0.0 and rep["mean_abs"] <= rep["max_abs"]


def test_bf16_workload_meets_the_reported_bounds(oracle_mod):
    w = Workload(3, "W4-bf16-small", 4, BF16, 1 << 16, "outliers", (Q4,), (2,))
    host = w.inputs()
    out, _ = oracle_mod.allreduce(BF16, Q4, 2, host)
    assert bench.error_vs_exact(host, out, BF16, Q4, 2)["within_bound_fraction"] == 1.0


@pytest.mark.parametrize("fmt,stages", [(FP, 1), (Q4, 2)])
def test_a_planted_error_is_reported(oracle_mod, fmt, stages):
    wl = sweep_workload(1 << 16)
    host = wl.inputs()
    out, _ = oracle_mod.allreduce(wl.dtype, fmt, stages, host)
    vals = out.view(np.float16).astype(np.float32)
    vals[100] += 4.0  # far beyond 1 ulp and beyond any block's scale bound
    bad = to_bits(vals, F16)
    rep = bench.error_vs_exact(host, bad, wl.dtype, fmt, stages)
    assert rep["within_bound_fraction"] < 1.0
    assert rep["max_abs"] >= 3.0


def test_per_recipe_oracle_timing_covers_every_workload():
    res = bench.oracle_per_config(threads=2, m=1 << 12)
    assert len(res) == len(workloads())
    for w, (name, row) in zip(workloads().values(), res.items()):
        assert name.startswith(w.name)
        assert len(row) == len(w.formats) * len(w.stages)
        assert all(v > 0 for v in row.values())
