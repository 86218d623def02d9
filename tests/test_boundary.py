"""The C ABI boundary, without a GPU: the library builds and loads, exports
every function include/qr.h declares, agrees with the oracle's header and
the quick_all_reduce page on enum values and encoded sizes, and rejects bad
arguments on the host before any CUDA call."""
import ctypes
import json
import os
import re

import pytest

import quantized_allreduce_codec_gb300 as qr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from quantized_allreduce_codec_gb300 import build
    build.build()
    return qr.lib()


def header_functions(path):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qr_[a-z0-9_]+)\s*\(", text)))


def header_enum(path, prefix):
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    return {k: int(v) for k, v in re.findall(rf"\b({prefix}[A-Z0-9_]+)\s*=\s*(\d+)", text)}


def test_exports_every_declared_function(L):
    names = header_functions(os.path.join(ROOT, "include", "qr.h"))
    assert set(names) == set(qr.EXPORTS)
    for name in names:
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {qr.LIB_PATH}").read()
    for name in names:
        assert re.search(rf"\bT {name}\b", out), name


def test_enums_agree_with_oracle_and_page():
    lib_fmt = header_enum(os.path.join(ROOT, "include", "qr.h"), "QR_")
    orc = header_enum(os.path.join(ROOT, "oracle", "qro.h"), "QRO_")
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "quick_reduce_regime.json")))
    reg = g["QuickReduceRegime"]
    assert lib_fmt["QR_FP"] == reg["FP"] == orc["QRO_FP"]
    assert lib_fmt["QR_Q8"] == reg["INT8"] == orc["QRO_Q8"]
    assert lib_fmt["QR_Q6"] == reg["INT6"] == orc["QRO_Q6"]
    assert lib_fmt["QR_Q4"] == reg["INT4"] == orc["QRO_Q4"]
    assert lib_fmt["QR_FP8"] == orc["QRO_FP8"]
    assert lib_fmt["QR_Q8_ASYM"] == orc["QRO_Q8A"]
    assert lib_fmt["QR_Q4_ASYM"] == orc["QRO_Q4A"]
    assert lib_fmt["QR_F16"] == orc["QRO_F16"] and lib_fmt["QR_BF16"] == orc["QRO_BF16"]
    assert lib_fmt["QR_BF16_AS_F16"] == orc["QRO_BF16_AS_F16"]
    for name, v in lib_fmt.items():
        if name.startswith("QR_ERR") or name == "QR_OK":
            assert qr.STATUS[v] == name


@pytest.mark.parametrize("fmt", range(7))
@pytest.mark.parametrize("n", [0, 8, 32, 40, 8192, 8200, 1 << 20])
def test_encoded_bytes_match_oracle(L, oracle_mod, fmt, n):
    assert qr.qr_encoded_bytes(fmt, n) == oracle_mod.encoded_bytes(fmt, n)


def test_encoded_bytes_table():
    # bytes per 32-element block: codes + fp16 scale (+ fp16 zero-point)
    per_block = {qr.QR_Q8: 34, qr.QR_FP8: 34, qr.QR_Q6: 26, qr.QR_Q4: 18,
                 qr.QR_Q8_ASYM: 36, qr.QR_Q4_ASYM: 20}
    for f, b in per_block.items():
        assert qr.qr_encoded_bytes(f, 32 * 1000) == 1000 * b
    assert qr.qr_encoded_bytes(qr.QR_FP, 1000) == 2000
    assert qr.qr_encoded_bytes(9, 1000) == 0


def test_kernel_path_follows_the_tables(L):
    from select_table_util import expected_path, limits, parse_tables
    tabs = parse_tables()
    assert qr.qr_forced_kernel_path() == qr.PATH_TABLE  # the tables route by default
    shapes = [(1, dt, fmt, 0) for dt in (0, 1) for fmt in range(7)]
    shapes += [(W, dt, fmt, st) for W in (1, 2, 4, 8) for dt in (0, 1, 2) for fmt in range(7) for st in (1, 2)]
    for W, dt, fmt, st in shapes:
        l1, l2 = limits(tabs, W, dt, fmt, st)
        assert l1 <= l2
        for n in {8, l1, l1 + 8, l2, l2 + 8, qr.MAX_ELEMS}:
            n = max(8, min(n, qr.MAX_ELEMS))
            assert qr.qr_kernel_path(W, dt, fmt, st, n) == expected_path(tabs, W, dt, fmt, st, n), (W, dt, fmt, st, n)
    # shapes no call can have
    assert qr.qr_kernel_path(2, 2, 1, 0, 64) == -1   # the cast option has no encode-only call
    assert qr.qr_kernel_path(3, 0, 1, 2, 64) == -1
    assert qr.qr_kernel_path(2, 0, 7, 2, 64) == -1
    assert qr.qr_kernel_path(2, 0, 1, 3, 64) == -1
    assert qr.qr_kernel_path(2, 5, 1, 2, 64) == -1


def test_forced_path_is_process_wide_and_reversible(L):
    old = qr.qr_forced_kernel_path()
    try:
        for path in (qr.PATH_DIRECT, qr.PATH_PIPELINE_NARROW, qr.PATH_PIPELINE):
            qr.qr_set_kernel_path(path)
            assert qr.qr_forced_kernel_path() == path
            for W, dt, fmt, st, n in ((2, 0, 1, 2, 64), (8, 1, 6, 1, 1 << 30), (1, 0, 3, 0, 4096)):
                assert qr.qr_kernel_path(W, dt, fmt, st, n) == path
        with pytest.raises(qr.QRError, match="QR_ERR_PATH"):
            qr.qr_set_kernel_path(3)
        assert qr.qr_forced_kernel_path() == qr.PATH_PIPELINE   # unchanged by the refused value
        with qr.forced_kernel_path(qr.PATH_DIRECT):
            assert qr.qr_forced_kernel_path() == qr.PATH_DIRECT
        assert qr.qr_forced_kernel_path() == qr.PATH_PIPELINE
        qr.qr_set_kernel_path(qr.PATH_TABLE)
        from select_table_util import expected_path, parse_tables
        assert qr.qr_kernel_path(8, 0, 3, 1, 8192 * 8192) == expected_path(parse_tables(), 8, 0, 3, 1, 8192 * 8192)
    finally:
        qr.qr_set_kernel_path(old)
    assert qr.qr_forced_kernel_path() == old


def test_status_strings(L):
    for s in range(len(qr.STATUS)):
        assert qr.qr_status_string(s)
    assert qr.qr_status_string(99) == "unknown status"


# Host-side validation: fake, never dereferenced addresses.
A, B, C = 0x10000, 0x200000, 0x4000000


def _ar(W, dt, fmt, stages, inputs, n, out, wire=None):
    arr = (ctypes.c_void_p * max(len(inputs), 1))(*inputs)
    return qr.lib().qr_allreduce_emulated(W, dt, fmt, stages, ctypes.cast(arr, ctypes.c_void_p), n,
                                          out, wire, None)


def test_allreduce_argument_errors(L):
    ok_in = [A, B]
    assert _ar(2, 0, 1, 2, ok_in, 0, None) == 0                      # empty message: nothing to do
    assert _ar(2, 0, 1, 2, ok_in, 64, None) == 1                     # QR_ERR_NULL
    assert _ar(2, 0, 1, 2, [A, 0], 64, C) == 1                       # NULL rank pointer
    assert _ar(2, 3, 1, 2, ok_in, 64, C) == 2                        # QR_ERR_DTYPE
    assert _ar(2, 0, 7, 2, ok_in, 64, C) == 3                        # QR_ERR_FORMAT
    assert _ar(3, 0, 1, 2, [A, B, A], 64, C) == 4                    # QR_ERR_WORLD
    assert _ar(16, 0, 1, 2, ok_in * 8, 64, C) == 4
    assert _ar(2, 0, 1, 3, ok_in, 64, C) == 5                        # QR_ERR_STAGES
    assert _ar(2, 0, 1, 1, ok_in, 64, C, C + (1 << 20)) == 5         # wire with one stage
    assert _ar(2, 0, 1, 2, ok_in, 60, C) == 6                        # 120 bytes: not % 16
    assert _ar(2, 0, 1, 2, ok_in, (1 << 36) + 8, C) == 6             # too large
    assert _ar(2, 0, 1, 2, [A + 2, B], 64, C) == 7                   # QR_ERR_ALIGN
    assert _ar(2, 0, 1, 2, ok_in, 64, C + 8) == 7
    assert _ar(2, 0, 1, 2, ok_in, 64, C, C + (1 << 20) + 4) == 7
    assert _ar(2, 0, 1, 2, ok_in, 64, A + 64) == 8                   # out overlaps an input
    assert _ar(2, 0, 1, 2, ok_in, 64, C, B + 16) == 8                # wire overlaps an input
    assert _ar(2, 0, 1, 2, ok_in, 64, C, C + 64) == 8                # wire overlaps out


def test_codec_argument_errors(L):
    q, d = qr.lib().qr_quantize, qr.lib().qr_dequantize
    assert q(0, 1, A, 0, None, None) == 0
    assert q(0, 1, None, 64, B, None) == 1
    assert q(5, 1, A, 64, B, None) == 2
    assert q(0, 8, A, 64, B, None) == 3
    assert q(0, 1, A, 12, B, None) == 6
    assert q(0, 1, A + 8, 64, B, None) == 7
    assert q(0, 1, A, 64, A + 16, None) == 8
    assert d(0, 1, A, 64, None, None) == 1
    assert d(1, 4, A, 64, A + 32, None) == 8
    assert d(0, 2, A, 64, B + 2, None) == 7
    assert q(2, 1, A, 64, B, None) == 2                               # cast option: allreduce only
    assert d(2, 1, A, 64, B, None) == 2
    assert qr.lib().qr_selftest_wait_timeout(0, None) == 6           # limit out of range
    assert qr.lib().qr_selftest_wait_timeout(1000001, None) == 6
    assert qr.lib().qr_selftest_reciprocal(None, None) == 1         # no buffer
    assert qr.lib().qr_selftest_reciprocal(A + 4, None) == 7         # misaligned


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(qr, "_lib", None)
    monkeypatch.setattr(qr, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        qr.lib()


def test_stage1_bytes_geometry(L):
    # W x W slots of ceil(nb / W) blocks each, padded to 16 bytes
    for W in (1, 2, 4, 8):
        for fmt, per_block in ((1, 34), (2, 26), (3, 18), (4, 34), (5, 36), (6, 20), (0, 64)):
            for n in (8, 40, 8200, 1 << 20):
                nb = (n + 31) // 32
                cnb = (nb + W - 1) // W
                assert qr.qr_stage1_bytes(W, fmt, n) == W * W * ((cnb * per_block + 15) // 16 * 16)
    assert qr.qr_stage1_bytes(3, 1, 64) == 0
    assert qr.qr_stage1_bytes(2, 9, 64) == 0


def test_host_workspace_bytes_geometry(L):
    # two chunk buffers of W inputs + output + payload, each region padded to 256 bytes
    pad = lambda b: (b + 255) // 256 * 256  # noqa: E731
    for W in (1, 2, 4, 8):
        for fmt in range(7):
            for chunk in (32, 8192, 1 << 21, (1 << 21) + 96):
                want = 2 * ((W + 1) * pad(chunk * 2) + pad(qr.qr_encoded_bytes(fmt, chunk)))
                assert qr.qr_host_workspace_bytes(W, fmt, chunk) == want
    assert qr.qr_host_workspace_bytes(2, 1, 0) == 0       # chunk of 0
    assert qr.qr_host_workspace_bytes(2, 1, 48) == 0      # not whole blocks
    assert qr.qr_host_workspace_bytes(3, 1, 64) == 0      # W
    assert qr.qr_host_workspace_bytes(2, 7, 64) == 0      # format


def _host(W, dt, fmt, stages, inputs, n, out, wire, ws, ws_bytes, chunk):
    arr = (ctypes.c_void_p * max(len(inputs), 1))(*inputs)
    return qr.lib().qr_allreduce_host(W, dt, fmt, stages, ctypes.cast(arr, ctypes.c_void_p), n, out, wire,
                                      ws, ws_bytes, chunk, None)


def test_host_entry_argument_errors(L):
    # host buffers need no alignment; every check runs before any CUDA call
    ha, hb, hc = 0x10000001, 0x20000003, 0x30000005
    chunk = 1 << 12
    need = qr.qr_host_workspace_bytes(2, 1, chunk)
    ok = dict(ws=C, ws_bytes=need, chunk=chunk)
    assert _host(2, 0, 1, 2, [ha, hb], 0, None, None, **ok) == 0            # empty message
    assert _host(2, 0, 1, 2, [ha, hb], 64, None, None, **ok) == 1           # QR_ERR_NULL (out)
    assert _host(2, 0, 1, 2, [ha, 0], 64, hc, None, **ok) == 1              # NULL rank pointer
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, None, None, need, chunk) == 1  # no workspace
    assert _host(2, 3, 1, 2, [ha, hb], 64, hc, None, **ok) == 2             # QR_ERR_DTYPE
    assert _host(2, 0, 9, 2, [ha, hb], 64, hc, None, **ok) == 3             # QR_ERR_FORMAT
    assert _host(3, 0, 1, 2, [ha, hb, ha], 64, hc, None, **ok) == 4         # QR_ERR_WORLD
    assert _host(2, 0, 1, 1, [ha, hb], 64, hc, hc + (1 << 20), **ok) == 5   # wire with one stage
    assert _host(2, 0, 1, 2, [ha, hb], 60, hc, None, **ok) == 6             # not % 16 bytes
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, None, C, need - 1, chunk) == 6  # workspace too small
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, None, C, need, 40) == 6      # chunk not whole blocks
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, None, C + 8, need, chunk) == 7  # workspace alignment
    assert _host(2, 0, 1, 2, [ha, hb], 64, ha + 100, None, **ok) == 8       # out overlaps an input
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, hb + 2, **ok) == 8           # wire overlaps an input
    assert _host(2, 0, 1, 2, [ha, hb], 64, hc, hc + 64, **ok) == 8          # wire overlaps out


def test_noalloc_scratch_size_agrees_with_header():
    text = open(os.path.join(ROOT, "include", "qr.h")).read()
    m = re.search(r"#define\s+QR_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "QR_NOALLOC_SCRATCH_BYTES not found in include/qr.h"
    assert qr.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def _staged(W, dt, fmt, inputs, n, out, wire, stage1):
    arr = (ctypes.c_void_p * max(len(inputs), 1))(*inputs)
    return qr.lib().qr_allreduce_staged(W, dt, fmt, ctypes.cast(arr, ctypes.c_void_p), n, out, wire, stage1, None)


def _noalloc(W, dt, fmt, inputs, n, out, wire):
    arr = (ctypes.c_void_p * max(len(inputs), 1))(*inputs)
    return qr.lib().qr_allreduce_staged_noalloc(W, dt, fmt, ctypes.cast(arr, ctypes.c_void_p), n, out, wire, None)


def test_staged_entries_share_argument_checks(L):
    # both staged entry points validate the same way; the one without a
    # stage-1 argument adds the bound on its built-in array.  Every case
    # below is refused on the host, before any CUDA call.
    D = 0x8000000
    ok_in = [A, B]
    for call in (lambda *a: _staged(*a, D), _noalloc):
        assert call(2, 0, 1, ok_in, 0, None, None) == 0                  # empty message
        assert call(2, 0, 1, ok_in, 64, C, None) == 1                    # no wire
        assert call(2, 0, 1, [A, 0], 64, C, C + 4096) == 1              # NULL rank pointer
        assert call(2, 3, 1, ok_in, 64, C, C + 4096) == 2               # dtype (no cast option here)
        assert call(2, 2, 1, ok_in, 64, C, C + 4096) == 2
        assert call(2, 0, 7, ok_in, 64, C, C + 4096) == 3               # format
        assert call(3, 0, 1, [A, B, A], 64, C, C + 4096) == 4           # W
        assert call(2, 0, 1, ok_in, 60, C, C + 4096) == 6               # not % 16 bytes
        assert call(2, 0, 1, [A + 2, B], 64, C, C + 4096) == 7          # alignment
        assert call(2, 0, 1, ok_in, 64, C, C + 4100) == 7
        assert call(2, 0, 1, ok_in, 64, A + 64, C + 4096) == 8          # out overlaps an input
        assert call(2, 0, 1, ok_in, 64, C, C + 64) == 8                 # wire overlaps out
    assert _staged(2, 0, 1, ok_in, 64, C, C + 4096, None) == 1          # no stage-1 buffer
    assert _staged(2, 0, 1, ok_in, 64, C, C + 4096, D + 8) == 7         # stage-1 alignment
    assert _staged(2, 0, 1, ok_in, 64, C, C + 4096, C + 32) == 8        # stage 1 overlaps out
    n = 8 << 20  # W=2 Q8: about 17.8 MB of stage-1 space, beyond the built-in array
    assert qr.qr_stage1_bytes(2, 1, n) > qr.NOALLOC_SCRATCH_BYTES
    assert _noalloc(2, 0, 1, ok_in, n, C, C + (64 << 20)) == 11          # QR_ERR_SCRATCH


def test_wrappers_refuse_a_rank_list_of_the_wrong_length(L):
    # the C side reads exactly W pointers; the binding never hands it fewer
    with pytest.raises(ValueError, match="rank buffers"):
        qr.qr_allreduce_emulated(2, qr.F16, qr.QR_Q8, 2, [A], 64, C)
    with pytest.raises(ValueError, match="rank buffers"):
        qr.qr_allreduce_staged(4, qr.F16, qr.QR_Q8, [A, B], 64, C, C + 4096, 0x8000000)
    with pytest.raises(ValueError, match="rank buffers"):
        qr.qr_allreduce_staged_noalloc(8, qr.F16, qr.QR_Q8, [A, B, C], 64, C, C + 4096)
    with pytest.raises(ValueError, match="rank buffers"):
        qr.qr_allreduce_host(2, qr.F16, qr.QR_Q8, 2, [A, B, C], 64, C, None, workspace=0x8000000,
                             workspace_bytes=1 << 30)
