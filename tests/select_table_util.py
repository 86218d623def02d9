"""The generated kernel-path tables as the tests read them: parsed from
csrc/qr_select_table.h, and the path they give a call (direct up to the
direct limit, narrow tiles up to the narrow-tile limit, wide tiles beyond;
narrow tiles exist for W <= 4 only)."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "quantized_allreduce_codec_gb300", "csrc", "qr_select_table.h")
WORLDS = (1, 2, 4, 8)
DIRECT, NARROW, WIDE = 0, 1, 2


def parse_tables():
    """{name: nested [dt][mode][w][fmt] list} for kDirectLimitTable and
    kNarrowTileLimitTable."""
    text = open(HEADER).read()
    out = {}
    for name in ("kDirectLimitTable", "kNarrowTileLimitTable"):
        body = text[text.index(name + "[3][3][4][7] = {"):]  # the definition, not a mention in a comment
        body = body[:body.index("};")]
        vals = [int(v) for v in re.findall(r"(\d+)ull", body)]
        assert len(vals) == 3 * 3 * 4 * 7, name
        out[name] = [[[vals[((d * 3 + m) * 4 + w) * 7:((d * 3 + m) * 4 + w) * 7 + 7] for w in range(4)]
                      for m in range(3)] for d in range(3)]
    return out


def limits(tabs, W, dt, fmt, stages):
    """(direct limit, narrow-tile limit) of a call shape (stages 0: encode-only)."""
    w = 0 if stages == 0 else WORLDS.index(W)
    return tabs["kDirectLimitTable"][dt][stages][w][fmt], tabs["kNarrowTileLimitTable"][dt][stages][w][fmt]


def expected_path(tabs, W, dt, fmt, stages, n):
    l1, l2 = limits(tabs, W, dt, fmt, stages)
    if n <= l1:
        return DIRECT
    if n <= l2:
        return NARROW
    return WIDE
