"""GPU parity: libqr.so (through the C ABI) against the CPU oracle.

Codes, scales, zero-points and outputs must agree bit for bit.  Small and
ragged sizes are compared element by element over the whole message (sizes
span several 8192-element tiles plus a partial final block); the five
workloads run at full size in the bench's launch configuration and are
compared on sampled blocks, which the oracle computes one block at a time.
"""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import (ALL_FORMATS, BF16, F16, FP, FP8, Q4, Q4A, Q6,
                                                    Q8, Q8A, from_bits, sweep_workload, to_bits,
                                                    workloads)
from qr_gpu_util import (dev_u16, gather_blocks, gpu_allreduce, gpu_dequantize, gpu_quantize,
                         out_buffer, sample_blocks, split_encoded)

pytestmark = pytest.mark.gpu

QUANT = (FP8, Q8, Q6, Q4, Q8A, Q4A)
SMALL_SIZES = [8, 24, 32, 40, 4096, 8192, 8200, 3 * 8192 + 40]


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qr.lib()
    qr.qr_device_error(clear=True)
    yield
    assert qr.qr_device_error(clear=True) == 0, "a kernel raised its wait-limit flag"


@pytest.fixture(params=["direct", "pipeline", "pipeline_narrow"])
def path(request):
    """Run the test once through each kernel: the direct (small-message)
    kernel and the bulk-copy pipeline with wide and with narrow tiles."""
    forced = {"direct": qr.PATH_DIRECT, "pipeline": qr.PATH_PIPELINE,
              "pipeline_narrow": qr.PATH_PIPELINE_NARROW}[request.param]
    with qr.forced_kernel_path(forced):
        yield request.param


def spread_values(rng, n, dtype, zero_blocks=True):
    """N(0,1) with per-block magnitudes from 2^-20 to 2^12 (bf16: to 2^40),
    a few all-zero and constant blocks, and some negative zeros."""
    nb = (n + 31) // 32
    hi = 12 if dtype == F16 else 40
    mags = np.exp2(rng.uniform(-20, hi, nb)).astype(np.float32)
    x = (rng.standard_normal(n).astype(np.float32) * np.repeat(mags, 32)[:n]).astype(np.float32)
    if dtype == F16:
        x = np.clip(x, -60000, 60000)
    if zero_blocks and nb > 4:
        x[32:64] = 0.0
        x[64:96] = np.float32(1.5)        # constant block: asymmetric scale 0
        x[96:100] = -0.0
    return to_bits(x, dtype)


def assert_encoded_equal(got, want, fmt, n):
    if fmt == FP:
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
        return
    gc, gs, gz = split_encoded(got, fmt, n)
    wc, ws, wz = split_encoded(want, fmt, n)
    bad_scale = np.nonzero(gs != ws)[0]
    assert bad_scale.size == 0, f"scales differ at blocks {bad_scale[:8]}"
    if gz is not None:
        bad_z = np.nonzero(gz != wz)[0]
        assert bad_z.size == 0, f"zero-points differ at blocks {bad_z[:8]}"
    bad = np.nonzero(np.any(gc != wc, axis=1))[0]
    assert bad.size == 0, f"codes differ at blocks {bad[:8]}"


def assert_bits_equal(got, want, what="out"):
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements differ, first at {bad[:6]}: "
                           f"gpu {got[bad[:6]]} oracle {want[bad[:6]]}")


# ----------------------------------------------------------------------------
# codec
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("n", SMALL_SIZES)
@pytest.mark.parametrize("fmt", ALL_FORMATS)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_quantize_parity(oracle_mod, dtype, fmt, n, path):
    xb = spread_values(np.random.default_rng(1000 + n + 17 * fmt), n, dtype)
    assert_encoded_equal(gpu_quantize(dtype, fmt, xb), oracle_mod.quantize(dtype, fmt, xb), fmt, n)


@pytest.mark.parametrize("n", SMALL_SIZES)
@pytest.mark.parametrize("fmt", ALL_FORMATS)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_dequantize_parity(oracle_mod, dtype, fmt, n):
    xb = spread_values(np.random.default_rng(2000 + n + 17 * fmt), n, dtype)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    assert_bits_equal(gpu_dequantize(dtype, fmt, enc, n), oracle_mod.dequantize(dtype, fmt, enc, n))


@pytest.mark.parametrize("fmt", QUANT)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_dequantize_arbitrary_codes(oracle_mod, dtype, fmt):
    """Every code pattern the layout can hold (also ones the encoder never
    emits), under random fp16 scales and zero-points."""
    rng = np.random.default_rng(3000 + fmt)
    n = 32 * 2048
    enc = rng.integers(0, 256, qr.qr_encoded_bytes(fmt, n), dtype=np.uint8)
    codes, scales, zps = split_encoded(enc, fmt, n)
    scales[:] = to_bits(np.exp2(rng.uniform(-20, 4, scales.size)).astype(np.float32), F16)
    if zps is not None:
        zps[:] = to_bits(rng.uniform(-100, 100, zps.size).astype(np.float32), F16)
    if fmt == FP8:  # NaN codes are outside the contract
        codes[(codes & 0x7F) == 0x7F] = 0x7E
    assert_bits_equal(gpu_dequantize(dtype, fmt, enc, n), oracle_mod.dequantize(dtype, fmt, enc, n))


# ----------------------------------------------------------------------------
# allreduce, whole-message comparison
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("n", [8, 40, 8200, 3 * 8192 + 40])
@pytest.mark.parametrize("stages", [1, 2])
@pytest.mark.parametrize("fmt", ALL_FORMATS)
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("W", [1, 2, 4, 8])
def test_allreduce_parity(oracle_mod, W, dtype, fmt, stages, n, path):
    rng = np.random.default_rng(4000 + 7 * W + 13 * fmt + n + stages)
    xs = [spread_values(rng, n, dtype, zero_blocks=(r == 0)) for r in range(W)]
    out, wire = gpu_allreduce(dtype, fmt, stages, xs)
    o_out, o_wire = oracle_mod.allreduce(dtype, fmt, stages, xs)
    assert_bits_equal(out, o_out)
    if stages == 2:
        assert_encoded_equal(wire, o_wire, fmt, n)


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("fmt", [Q8A, Q4A, Q8, Q4])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_offset_blocks_parity(oracle_mod, W, dtype, fmt, path):
    """Blocks far from zero with small ranges (+-500 + 0.3 N(0,1) per rank):
    the sums' fp16 zero-points lie many steps above their minima, so the
    asymmetric requantization must clamp codes at 0 (the clamp-free fast
    path must not be taken); the symmetric formats get scales set by large,
    nearly equal magnitudes."""
    rng = np.random.default_rng(7000 + 11 * W + fmt + 3 * dtype)
    n = 3 * 8192 + 40
    sign = np.repeat(rng.choice(np.array([-1.0, 1.0], np.float32), (n + 31) // 32), 32)[:n]
    xs = [to_bits((sign * 500.0 + 0.3 * rng.standard_normal(n)).astype(np.float32), dtype)
          for _ in range(W)]
    for stages in (1, 2):
        out, wire = gpu_allreduce(dtype, fmt, stages, xs)
        o_out, o_wire = oracle_mod.allreduce(dtype, fmt, stages, xs)
        assert_bits_equal(out, o_out)
        if stages == 2:
            assert_encoded_equal(wire, o_wire, fmt, n)


@pytest.mark.parametrize("fmt", ALL_FORMATS)
def test_allreduce_without_wire_gives_same_output(oracle_mod, fmt, path):
    rng = np.random.default_rng(5000 + fmt)
    n = 2 * 8192 + 24
    xs = [to_bits(rng.standard_normal(n).astype(np.float32), F16) for _ in range(4)]
    out_w, _ = gpu_allreduce(F16, fmt, 2, xs, want_wire=True)
    out_nw, _ = gpu_allreduce(F16, fmt, 2, xs, want_wire=False)
    assert_bits_equal(out_w, out_nw)


@pytest.mark.parametrize("fmt", [FP, Q8, Q6, Q4A])
def test_result_independent_of_tile_assignment(fmt, path):
    """Starting the same data 3 tiles + 5 blocks later (so every block lands
    on a different thread, rotation and CTA) gives the same blocks."""
    rng = np.random.default_rng(6000 + fmt)
    n = 16 * 8192
    xs = [to_bits(rng.standard_normal(n).astype(np.float32) * 3, BF16) for _ in range(2)]
    out, wire = gpu_allreduce(BF16, fmt, 2, xs)
    off = 3 * 8192 + 5 * 32
    dev = [dev_u16(x) for x in xs]
    sub = [t[off:] for t in dev]
    out2, wire2 = gpu_allreduce(BF16, fmt, 2, None, dev_inputs=sub)
    assert_bits_equal(out2, out[off:])
    if fmt != FP:
        c1, s1, z1 = split_encoded(wire, fmt, n)
        c2, s2, z2 = split_encoded(wire2, fmt, n - off)
        assert np.array_equal(c1[off // 32:], c2) and np.array_equal(s1[off // 32:], s2)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_degenerate_blocks(oracle_mod, dtype, path):
    """All-zero, constant, negative-zero, underflowing and (bf16) saturating
    blocks through every format and both stage counts."""
    n = 32 * 64
    x = np.zeros(n, np.float32)
    x[32:64] = -0.0
    x[64:96] = 7.25
    x[96:128] = -3.0
    x[128:160] = 2.0 ** -30
    x[160:192] = np.linspace(-1, 1, 32)
    x[192:224] = 1e-7 * np.arange(32)
    if dtype == BF16:
        x[224:256] = 1e30
        x[256:288] = np.linspace(-3e37, 3e37, 32)
    else:
        x[224:256] = 65504.0
        x[256:288] = np.linspace(-60000, 60000, 32)
    xs = [to_bits(x, dtype), to_bits(x[::-1].copy(), dtype)]
    for fmt in ALL_FORMATS:
        assert_encoded_equal(gpu_quantize(dtype, fmt, xs[0]), oracle_mod.quantize(dtype, fmt, xs[0]),
                             fmt, n)
        for stages in (1, 2):
            out, wire = gpu_allreduce(dtype, fmt, stages, xs)
            o_out, o_wire = oracle_mod.allreduce(dtype, fmt, stages, xs)
            assert_bits_equal(out, o_out)
            if stages == 2:
                assert_encoded_equal(wire, o_wire, fmt, n)


def test_empty_message_launches_nothing():
    x = torch.zeros(16, dtype=torch.float16, device="cuda")
    qr.qr_allreduce_emulated(2, F16, Q8, 2, [x, x], 0, x)
    qr.qr_quantize(F16, Q8, x, 0, x)
    qr.qr_dequantize(F16, Q8, x, 0, x)


def test_gpu_argument_errors():
    x = torch.zeros(64, dtype=torch.float16, device="cuda")
    y = torch.zeros(64, dtype=torch.float16, device="cuda")
    with pytest.raises(qr.QRError, match="QR_ERR_ALIGN"):
        qr.qr_allreduce_emulated(2, F16, Q8, 2, [x[1:].data_ptr(), y], 56, torch.empty_like(x))
    with pytest.raises(qr.QRError, match="QR_ERR_OVERLAP"):
        qr.qr_allreduce_emulated(2, F16, Q8, 2, [x, y], 64, x)
    with pytest.raises(qr.QRError, match="QR_ERR_WORLD"):
        qr.qr_allreduce_emulated(3, F16, Q8, 2, [x, y, y], 64, torch.empty_like(x))


# ----------------------------------------------------------------------------
# the five workloads at full size, sampled blocks
# ----------------------------------------------------------------------------
def check_sampled(oracle_mod, wl_dtype, fmt, stages, xs_host, out, wire, n, seed, count=3000):
    blocks = sample_blocks(n, count, seed)
    sub = [gather_blocks(x, blocks) for x in xs_host]
    o_out, o_wire = oracle_mod.allreduce(wl_dtype, fmt, stages, sub)
    assert_bits_equal(gather_blocks(out, blocks), o_out)
    if stages == 2 and wire is not None:
        if fmt == FP:
            assert_bits_equal(gather_blocks(wire.view(np.uint16), blocks), o_wire.view(np.uint16), "wire")
        else:
            gc, gs, gz = split_encoded(wire, fmt, n)
            wc, ws, wz = split_encoded(o_wire, fmt, sub[0].size)
            assert np.array_equal(gc[blocks], wc)
            assert np.array_equal(gs[blocks], ws)
            if gz is not None:
                assert np.array_equal(gz[blocks], wz)


def run_workload(oracle_mod, wl, fmts=None, stages_list=None, seed=0):
    """Sampled blocks against the oracle, plus a property that holds at any
    size: a second identical call gives the same bits everywhere (a pipeline
    race shows up as run-to-run differences)."""
    xs = wl.inputs()
    dev = [dev_u16(x) for x in xs]
    for fmt in fmts or wl.formats:
        for stages in stages_list or wl.stages:
            out, wire = gpu_allreduce(wl.dtype, fmt, stages, None, dev_inputs=dev)
            check_sampled(oracle_mod, wl.dtype, fmt, stages, xs, out, wire, wl.n, seed + fmt)
            out2, wire2 = gpu_allreduce(wl.dtype, fmt, stages, None, dev_inputs=dev)
            assert_bits_equal(out2, out, "repeat")
            if wire is not None:
                assert np.array_equal(wire2, wire)
    del dev
    torch.cuda.empty_cache()


def test_workload1_full_compare(oracle_mod):
    wl = workloads()[1]
    xs = wl.inputs()
    out, wire = gpu_allreduce(wl.dtype, Q8, 2, xs)
    o_out, o_wire = oracle_mod.allreduce(wl.dtype, Q8, 2, xs)
    assert_bits_equal(out, o_out)
    assert_encoded_equal(wire, o_wire, Q8, wl.n)


@pytest.mark.parametrize("size", [4096, 65536, 1 << 20, 16 << 20, 64 << 20])
def test_workload2_sweep_points(oracle_mod, size):
    wl = sweep_workload(size)
    run_workload(oracle_mod, wl, stages_list=(1, 2), seed=size)


def test_workload3(oracle_mod):
    run_workload(oracle_mod, workloads()[3], seed=3)


def test_workload4(oracle_mod):
    run_workload(oracle_mod, workloads()[4], seed=4)


def test_workload5(oracle_mod):
    run_workload(oracle_mod, workloads()[5], seed=5)


@pytest.mark.parametrize("fmt,stages", [(FP, 1), (Q8, 2), (Q4, 2)])
def test_full_compare_64MiB(oracle_mod, fmt, stages):
    """Every element of the tp2 table's largest message (W=2, fp16, 64 MiB
    per rank), in the bench's launch configuration, against the oracle,
    twice: a pipeline race would corrupt a few blocks anywhere."""
    wl = sweep_workload(64 << 20)
    xs = wl.inputs()
    dev = [dev_u16(x) for x in xs]
    o_out, o_wire = oracle_mod.allreduce(wl.dtype, fmt, stages, xs)
    for _ in range(2):
        out, wire = gpu_allreduce(wl.dtype, fmt, stages, None, dev_inputs=dev)
        assert_bits_equal(out, o_out)
        if stages == 2:
            assert_encoded_equal(wire, o_wire, fmt, wl.n)


def test_paths_agree_past_the_table_limits(oracle_mod):
    """By default the measured tables route every call shape; the three
    kernels give the same bits on a message just past a wide tile."""
    assert qr.qr_forced_kernel_path() == qr.PATH_TABLE
    rng = np.random.default_rng(7000)
    n = 4 * 1024 * 1024 + 8
    xs = [to_bits(rng.standard_normal(n).astype(np.float32), F16) for _ in range(2)]
    for fmt in (Q8, Q6, Q4A):
        res = []
        for path in (qr.PATH_PIPELINE, qr.PATH_DIRECT, qr.PATH_PIPELINE_NARROW):
            with qr.forced_kernel_path(path):
                res.append(gpu_allreduce(F16, fmt, 2, xs))
        for a, wa in res[1:]:
            assert_bits_equal(res[0][0], a, "paths")
            assert np.array_equal(res[0][1], wa)


@pytest.mark.parametrize("stages", [1, 2])
@pytest.mark.parametrize("dtype", [F16, BF16, qr.BF16_AS_F16])
@pytest.mark.parametrize("fmt", [Q8, Q6, Q4, Q8A, Q4A])
@pytest.mark.parametrize("W", [2, 4])
def test_block_kernel_parity(oracle_mod, W, dtype, fmt, stages):
    """The direct path of a W=2 or W=4 call of an integer format runs the
    block kernel from 3M (W=2) or 4M (W=4) elements per rank: a message just
    past that size with a ragged tail gives the same bits as the wide-tile
    pipeline (output and payload) and, on sampled blocks, as the oracle
    (fp16, bf16 and bf16 through fp16; the values stay inside the fp16
    range, as the cast option requires)."""
    rng = np.random.default_rng(7100 + 10 * W + fmt + 100 * int(dtype) + 1000 * stages)
    n = (4 << 20) + 40
    xs = []
    for _ in range(W):
        x = rng.standard_normal(n).astype(np.float32)
        x[rng.random(n) < 0.001] *= 50
        xs.append(to_bits(x, BF16 if dtype == qr.BF16_AS_F16 else dtype))  # the cast option takes bf16 messages
    with qr.forced_kernel_path(qr.PATH_DIRECT):
        out, wire = gpu_allreduce(dtype, fmt, stages, xs)
    with qr.forced_kernel_path(qr.PATH_PIPELINE):
        out_p, wire_p = gpu_allreduce(dtype, fmt, stages, xs)
    assert_bits_equal(out_p, out, "block kernel vs pipeline")
    if stages == 2:
        assert np.array_equal(wire_p, wire)
    blocks = sample_blocks(n, 600, 17 + fmt)
    sub = [np.concatenate([x[32 * b:32 * b + 32] for b in blocks]) for x in xs]
    o_out, _ = oracle_mod.allreduce(dtype, fmt, stages, sub)
    assert_bits_equal(np.concatenate([out[32 * b:32 * b + 32] for b in blocks]), o_out, "block kernel vs oracle")


@pytest.mark.parametrize("n", [40, 8200, 3 * 8192 + 40])
@pytest.mark.parametrize("stages", [1, 2])
@pytest.mark.parametrize("fmt", ALL_FORMATS)
@pytest.mark.parametrize("W", [1, 2, 8])
def test_bf16_cast_option_parity(oracle_mod, W, fmt, stages, n, path):
    """bf16 messages through the fp16 path (the cast option), inside the fp16
    range, against the oracle's reading of the option."""
    rng = np.random.default_rng(9500 + 7 * W + 13 * fmt + n + stages)
    xs = []
    for r in range(W):
        v = from_bits(spread_values(rng, n, F16, zero_blocks=(r == 0)), F16)
        xs.append(to_bits(v, BF16))
    out, wire = gpu_allreduce(qr.BF16_AS_F16, fmt, stages, xs)
    o_out, o_wire = oracle_mod.allreduce(qr.BF16_AS_F16, fmt, stages, xs)
    assert_bits_equal(out, o_out)
    if stages == 2:
        assert_encoded_equal(wire, o_wire, fmt, n)
