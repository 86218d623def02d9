"""Kernel-path selection table: from a measured sweep to csrc/qr_select_table.h.

Every qr_quantize and qr_allreduce_emulated call is served by one of three
kernels that compute identical bits: the direct kernel (one memory round
trip, lowest latency), the persistent bulk-copy pipeline with narrow (8 KiB)
tiles and the same pipeline with wide (16 KiB) tiles (highest bandwidth).
Which is fastest at a given message size depends on the call's shape --
dtype, stage mode (encode-only, one-stage, two-stage), rank count W and
format -- so the library routes by two per-shape size limits: messages of at
most the direct limit (elements per rank) take the direct kernel, those of at
most the narrow-tile limit the narrow-tile pipeline, longer ones the
wide-tile pipeline.  This is the GB300
counterpart of the per-(dtype, world size) size thresholds that the vLLM
quick_all_reduce page keeps in _QR_MIN_SIZE, and of the size rule in vLLM PR
#18473's description (custom allreduce for small messages, quick allreduce
above), applied to the choice this one-GPU data path actually has.

The sweep (``python bench.py --select-sweep OUT.json``) times the kernels at
every size of a grid for every shape; this module picks, per shape, the pair
of limits that minimises the summed relative excess time over the grid, and
writes the tables as a C header that libqr.so compiles in.  Usage:

    python -m quantized_allreduce_codec_gb300.select_table [SWEEP.json]

(default: select_sweep.json next to this file, the committed GB300 sweep).
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SWEEP = os.path.join(HERE, "select_sweep.json")
HEADER = os.path.join(HERE, "csrc", "qr_select_table.h")

MAX_ELEMS = 1 << 36         # QR_MAX_ELEMS: a limit this large means "always the direct kernel"
DTYPES = (0, 1, 2)          # fp16, bf16, bf16 through fp16 (allreduce only)
MODES = (0, 1, 2)           # encode-only (qr_quantize), one-stage, two-stage
WORLDS = (1, 2, 4, 8)
FORMATS = tuple(range(7))
DEFAULT_LIMIT = 4 << 20     # shapes the sweep does not cover


def valid_shape(dt: int, mode: int, W: int) -> bool:
    if mode == 0:
        return W == 1 and dt in (0, 1)
    return True


def choose_limits(points) -> tuple:
    """points: [(n, t_direct, t_narrow, t_wide)] over a size grid (t_narrow
    None where the narrow-tile pipeline was not measured).  The limits
    (L1, L2), L1 <= L2, among 0 and the grid sizes -- n <= L1: direct; n <= L2:
    narrow tiles; else wide tiles -- that minimise the sum over the grid of
    t_routed / t_best - 1; ties go to the smaller limits.  A limit at the
    largest size measured means that path won there too: it is extended to
    every size."""
    pts = sorted(points)
    narrow = all(p[2] is not None for p in pts)
    cands = [0] + [p[0] for p in pts]
    best = None
    for L1 in cands:
        for L2 in (cands if narrow else [L1]):
            if L2 < L1:
                continue
            cost = 0.0
            for n, td, tn, tw in pts:
                t = td if n <= L1 else tn if n <= L2 else tw
                cost += t / min(x for x in (td, tn, tw) if x is not None) - 1.0
            if best is None or cost < best[0] - 1e-12:
                best = (cost, L1, L2)
    _, L1, L2 = best if best else (0.0, 0, 0)
    top = pts[-1][0] if pts else None
    if L1 == top:
        L1 = L2 = MAX_ELEMS
    elif L2 == top:
        L2 = MAX_ELEMS
    return L1, L2


def choose_limit(points) -> int:
    """The direct limit alone, for points [(n, t_direct, t_pipeline)]."""
    return choose_limits([(n, td, None, tp) for n, td, tp in points])[0]


def records_of(data: dict) -> list:
    """The sweep's records as dicts (the committed file stores rows under
    `columns`; bench.py writes dicts)."""
    cols = data.get("columns")
    return [dict(zip(cols, r)) for r in data["records"]] if cols else data["records"]


def limits_from_sweep(records) -> dict:
    """{(dt, mode, W, fmt): (direct limit, narrow-tile limit)} from the sweep's records."""
    by_shape = {}
    for r in records:
        key = (r["dt"], r["mode"], r["W"], r["fmt"])
        by_shape.setdefault(key, []).append((r["n"], r["us_direct"], r.get("us_narrow"), r["us_pipeline"]))
    return {k: choose_limits(v) for k, v in by_shape.items()}


def table(limits: dict, which: int = 0) -> list:
    """The 3 x 3 x 4 x 7 nested list of limit `which` (0: direct, 1: narrow
    tiles) compiled into the library (0 for shapes no call can have)."""
    out = []
    for dt in DTYPES:
        a = []
        for mode in MODES:
            b = []
            for W in WORLDS:
                row = []
                for fmt in FORMATS:
                    if not valid_shape(dt, mode, W):
                        row.append(0)
                    else:
                        row.append(int(limits.get((dt, mode, W, fmt), (DEFAULT_LIMIT, DEFAULT_LIMIT))[which]))
                b.append(row)
            a.append(b)
        out.append(a)
    return out


def render(direct: list, narrow: list, source: str) -> str:
    lines = [
        "// qr_select_table.h -- kernel-path selection tables, GENERATED by",
        f"// quantized_allreduce_codec_gb300/select_table.py from {source}; do not edit.",
        "//",
        "// [dtype][mode][w][format]: messages of at most kDirectLimitTable elements",
        "// per rank take the direct kernel, those of at most kNarrowTileLimitTable",
        "// the narrow-tile pipeline, longer ones the wide-tile pipeline.  dtype:",
        "// fp16, bf16, bf16 through fp16; mode: encode-only (qr_quantize), one-stage,",
        "// two-stage; w: W = 1, 2, 4, 8; format: FP, Q8, Q6, Q4, FP8, Q8A, Q4A.  2^36",
        "// (the largest message) = every size; 0 for shapes no call can have.",
        "// Chosen per shape from the kernels' times over a size grid on GB300 (the",
        "// limits minimising the summed relative excess).",
        "#pragma once",
        "",
        "namespace qr {",
        "",
    ]
    dnames, mnames = ("fp16", "bf16", "bf16 through fp16"), ("encode", "one-stage", "two-stage")
    for name, tab in (("kDirectLimitTable", direct), ("kNarrowTileLimitTable", narrow)):
        lines.append(f"static constexpr unsigned long long {name}[3][3][4][7] = {{")
        for di, a in enumerate(tab):
            lines.append(f"    {{  // {dnames[di]}")
            for mi, b in enumerate(a):
                lines.append(f"        {{  // {mnames[mi]}")
                for wi, row in enumerate(b):
                    vals = ", ".join(f"{v}ull" for v in row)
                    lines.append(f"            {{{vals}}},  // W={WORLDS[wi]}")
                lines.append("        },")
            lines.append("    },")
        lines += ["};", ""]
    lines += ["}  // namespace qr", ""]
    return "\n".join(lines)


def generate(sweep_path: str = SWEEP) -> str:
    with open(sweep_path) as f:
        data = json.load(f)
    lim = limits_from_sweep(records_of(data))
    return render(table(lim, 0), table(lim, 1), os.path.basename(sweep_path))


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    path = argv[0] if argv else SWEEP
    text = generate(path)
    with open(HEADER, "w") as f:
        f.write(text)
    print(HEADER)


if __name__ == "__main__":
    main()
