"""Pins for the oracle's block codec (qr_quantize / qr_dequantize semantics).

The oracle encodes with rint and a clamp; these tests check it by other
routes: brute-force enumeration of every admissible code, blocks whose values
already sit on the quantization grid, a hand-worked block, independent bit
unpacking (Python integers), tail blocks, and error bounds.
"""
import numpy as np
import pytest
import torch

from quantized_allreduce_codec_gb300.inputs import (BF16, F16, FP, FP8, Q4, Q4A, Q6, Q8, Q8A,
                                                    from_bits, to_bits)

BITS = {Q8: 8, Q6: 6, Q4: 4, FP8: 8, Q8A: 8, Q4A: 4}
SYM = (Q8, Q6, Q4)
ASYM = (Q8A, Q4A)
QUANT = (FP8, Q8, Q6, Q4, Q8A, Q4A)


def f16val(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)


def fp16_sat(v32):
    return np.clip(np.float32(v32), -65504.0, 65504.0).astype(np.float16).astype(np.float32)


def e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()


def parse(enc, fmt, n):
    """Split an encoded message into per-block integer codes, scales, zps.

    Written independently of the oracle: the block's codes are read from a
    little-endian Python integer of the block's code bytes."""
    b = BITS[fmt]
    nb = (n + 31) // 32
    cb = 32 * b // 8
    codes = np.zeros((nb, 32), np.int64)
    for blk in range(nb):
        stream = int.from_bytes(bytes(enc[blk * cb:(blk + 1) * cb]), "little")
        for i in range(32):
            u = (stream >> (b * i)) & ((1 << b) - 1)
            if fmt in SYM and u >= (1 << (b - 1)):
                u -= 1 << b
            codes[blk, i] = u
    scales = f16val(enc[nb * cb:nb * cb + 2 * nb].view(np.uint16))
    zps = None
    if fmt in ASYM:
        zps = f16val(enc[nb * cb + 2 * nb:nb * cb + 4 * nb].view(np.uint16))
    return codes, scales, zps


def pick(dist, cands):
    """Index of the minimum distance; ties go to the even candidate."""
    best = dist.min()
    idx = np.nonzero(dist == best)[0]
    if len(idx) == 1:
        return cands[idx[0]]
    even = [cands[i] for i in idx if cands[i] % 2 == 0]
    assert len(even) == 1
    return even[0]


def random_blocks(rng, dtype, nblocks, spread=True):
    x = rng.standard_normal(nblocks * 32).astype(np.float32)
    if spread:  # magnitudes from 2^-20 to 2^12 across blocks
        x = x * np.repeat(np.exp2(rng.uniform(-20, 12, nblocks)).astype(np.float32), 32)
    return to_bits(x, dtype)


def with_saturating_blocks(rng, xb, dtype):
    """bf16 only: the last two blocks get magnitudes near 2^40 (one of them
    offset by 2^36 with a small spread), beyond what an fp16 scale or
    zero-point can hold, so the saturating fp16 rounding of the statistics
    decides the codes.  fp16 messages are returned unchanged."""
    if dtype != BF16:
        return xb
    x = from_bits(xb, dtype)
    x[-64:-32] = rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** 40)
    x[-32:] = np.float32(2.0 ** 36) + rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** 30)
    return to_bits(x, dtype)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("fmt", SYM)
def test_sym_codes_are_bruteforce_nearest(oracle_mod, dtype, fmt):
    rng = np.random.default_rng(100 + fmt)
    xb = with_saturating_blocks(rng, random_blocks(rng, dtype, 64), dtype)
    x = from_bits(xb, dtype)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    codes, scales, _ = parse(enc, fmt, x.size)
    Q = (1 << (BITS[fmt] - 1)) - 1
    cands = np.arange(-Q, Q + 1)
    for blk in range(64):
        xs = x[blk * 32:(blk + 1) * 32]
        a = np.max(np.abs(xs))
        assert scales[blk] == fp16_sat(np.float32(a) / np.float32(Q))
        if scales[blk] == 0:
            assert np.all(codes[blk] == 0)
            continue
        inv = np.float32(1.0) / np.float32(scales[blk])
        v = (xs * inv).astype(np.float32).astype(np.float64)
        for i in range(32):
            want = pick(np.abs(v[i] - cands), cands)
            assert codes[blk, i] == want, (blk, i, v[i])


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("fmt", ASYM)
def test_asym_codes_are_bruteforce_nearest(oracle_mod, dtype, fmt):
    rng = np.random.default_rng(200 + fmt)
    xb = with_saturating_blocks(rng, random_blocks(rng, dtype, 64), dtype)
    x = from_bits(xb, dtype)
    x[32:64] += np.float32(3.0)  # a block with a large offset
    xb = to_bits(x, dtype)
    x = from_bits(xb, dtype)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    codes, scales, zps = parse(enc, fmt, x.size)
    L = (1 << BITS[fmt]) - 1
    cands = np.arange(0, L + 1)
    for blk in range(64):
        xs = x[blk * 32:(blk + 1) * 32]
        m, M = np.min(xs), np.max(xs)
        assert scales[blk] == fp16_sat(np.float32(M - m) / np.float32(L))
        assert zps[blk] == fp16_sat(m)
        if scales[blk] == 0:
            assert np.all(codes[blk] == 0)
            continue
        inv = np.float32(1.0) / np.float32(scales[blk])
        v = ((xs - zps[blk]).astype(np.float32) * inv).astype(np.float32).astype(np.float64)
        for i in range(32):
            assert codes[blk, i] == pick(np.abs(v[i] - cands), cands), (blk, i)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_fp8_codes_are_bruteforce_nearest(oracle_mod, dtype):
    rng = np.random.default_rng(300)
    xb = with_saturating_blocks(rng, random_blocks(rng, dtype, 64), dtype)
    x = from_bits(xb, dtype)
    enc = oracle_mod.quantize(dtype, FP8, xb)
    codes, scales, _ = parse(enc, FP8, x.size)
    table = e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    for blk in range(64):
        xs = x[blk * 32:(blk + 1) * 32]
        a = np.max(np.abs(xs))
        assert scales[blk] == fp16_sat(np.float32(a) / np.float32(448.0))
        if scales[blk] == 0:
            assert np.all(codes[blk] == 0)
            continue
        inv = np.float32(1.0) / np.float32(scales[blk])
        v = (xs * inv).astype(np.float32).astype(np.float64)
        for i in range(32):
            vi = float(np.clip(v[i], -448.0, 448.0))
            dist = np.abs(vi - table[finite])
            best = dist.min()
            tied = [int(c) for c, d in zip(finite, dist) if d == best]
            if len(tied) > 1 and table[tied[0]] == 0.0:  # +0 / -0: keep the sign
                tied = [0x80] if np.signbit(v[i]) else [0x00]
            if len(tied) > 1:  # exact tie between two values: even significand
                tied = [c for c in tied if c % 2 == 0]
            assert len(tied) == 1
            assert codes[blk, i] == tied[0], (blk, i, v[i])


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("fmt", SYM)
def test_sym_grid_roundtrip(oracle_mod, dtype, fmt):
    """k * 2^e with some |k| = Qmax encodes to exactly k and decodes exactly."""
    rng = np.random.default_rng(400 + fmt)
    Q = (1 << (BITS[fmt] - 1)) - 1
    nblk = 24
    k = rng.integers(-Q, Q + 1, (nblk, 32))
    k[:, 0] = np.where(rng.random(nblk) < 0.5, Q, -Q)
    e = rng.integers(-12, 8, nblk)
    x = (k * np.exp2(e)[:, None]).astype(np.float32).reshape(-1)
    xb = to_bits(x, dtype)
    assert np.all(from_bits(xb, dtype) == x)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    codes, scales, _ = parse(enc, fmt, x.size)
    assert np.array_equal(codes, k)
    assert np.array_equal(scales, np.exp2(e).astype(np.float32))
    assert np.array_equal(oracle_mod.dequantize(dtype, fmt, enc, x.size), xb)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("fmt", ASYM)
def test_asym_grid_roundtrip(oracle_mod, dtype, fmt):
    """z + k * 2^e with k spanning 0..L encodes to exactly k."""
    rng = np.random.default_rng(500 + fmt)
    L = (1 << BITS[fmt]) - 1
    nblk = 24
    k = rng.integers(0, L + 1, (nblk, 32))
    k[:, 0], k[:, 1] = 0, L
    e = rng.integers(-10, -2, nblk)
    z = -np.exp2(e + 3) * rng.integers(1, 4, nblk)  # a few steps below zero, on the grid
    x = (z[:, None] + k * np.exp2(e)[:, None]).astype(np.float32).reshape(-1)
    xb = to_bits(x, dtype)
    ok = np.all(from_bits(xb, dtype).reshape(nblk, 32) == x.reshape(nblk, 32), axis=1)
    assert ok.sum() >= nblk // 2  # bf16 has 8 bits: keep the blocks that fit
    x = x.reshape(nblk, 32)[ok].reshape(-1)
    k = k[ok]
    xb = to_bits(x, dtype)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    codes, scales, zps = parse(enc, fmt, x.size)
    assert np.array_equal(codes, k)
    assert np.array_equal(scales, np.exp2(e[ok]).astype(np.float32))
    assert np.array_equal(zps, z[ok].astype(np.float32))
    assert np.array_equal(oracle_mod.dequantize(dtype, fmt, enc, x.size), xb)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_fp8_grid_roundtrip(oracle_mod, dtype):
    rng = np.random.default_rng(600)
    table = e4m3_table()
    nblk = 16
    # e4m3 codes with at most 4 significant bits fit both fp16 and bf16
    good = [c for c in range(256) if not np.isnan(table[c])]
    c = rng.choice(good, (nblk, 32))
    c[:, 0] = 0x7E  # 448 sets the scale exactly to 2^e
    e = rng.integers(-14, 4, nblk)
    x = (table[c] * np.exp2(e)[:, None]).astype(np.float32).reshape(-1)
    xb = to_bits(x, dtype)
    assert np.all(from_bits(xb, dtype) == x)
    enc = oracle_mod.quantize(dtype, FP8, xb)
    codes, scales, _ = parse(enc, FP8, x.size)
    # -0 and +0 are both exact encodings of a zero value
    same = (codes == c) | ((table[codes] == 0) & (table[c] == 0))
    assert np.all(same)
    assert np.array_equal(scales, np.exp2(e).astype(np.float32))
    assert np.array_equal(from_bits(oracle_mod.dequantize(dtype, FP8, enc, x.size), dtype), x)


def test_hand_worked_q8_block(oracle_mod):
    """One Q8 block worked by hand.

    x = [1, -0.5, 0.25, 2, 0, ...]: a = 2; 2/127 = 0.0157480315 rounds in
    fp16 to 2^-6 * (1 + 8/1024) = 0.0157470703125 (fp16 bits 0x2408);
    inv = 1/s = 63.5038759...; codes rint(x*inv) = 64, -32, 16, 127
    (127.0078 rounds to 127); decoded q*s = 1.0078125, -0.50390625,
    0.251953125, 1.9998779296875, and the last rounds to 2.0 in fp16
    (spacing 2^-10 on [1, 2))."""
    x = np.zeros(32, np.float32)
    x[:4] = [1.0, -0.5, 0.25, 2.0]
    enc = oracle_mod.quantize(F16, Q8, to_bits(x, F16))
    assert enc.size == 34
    assert list(enc[:4]) == [64, 256 - 32, 16, 127]
    assert np.all(enc[4:32] == 0)
    assert enc[32:34].view(np.uint16)[0] == 0x2408
    y = from_bits(oracle_mod.dequantize(F16, Q8, enc, 32), F16)
    assert list(y[:4]) == [1.0078125, -0.50390625, 0.251953125, 2.0]


def test_packing_known_answer_q6_q4(oracle_mod):
    """Q6 code i sits at bits [6i, 6i+6) of the little-endian block stream;
    Q4 byte j = (q_2j & 15) | (q_2j+1 & 15) << 4."""
    k6 = np.array([31, -31, 1, -1, 0, 17, -9, 5] * 4)
    x6 = (k6 * 0.25).astype(np.float32)
    enc = oracle_mod.quantize(F16, Q6, to_bits(x6, F16))
    stream = sum(((int(q) & 63) << (6 * i)) for i, q in enumerate(k6))
    assert bytes(enc[:24]) == stream.to_bytes(24, "little")
    # first four codes 31, -31 (=33), 1, -1 (=63) by hand:
    # bits: 011111 100001 000001 111111 -> bytes 0x5F, 0x18, 0xFC
    assert list(enc[:3]) == [0x5F, 0x18, 0xFC]
    k4 = np.array([7, -7, 3, -1] * 8)
    enc4 = oracle_mod.quantize(F16, Q4, to_bits((k4 * 0.5).astype(np.float32), F16))
    assert list(enc4[:2]) == [0x97, 0xF3]


@pytest.mark.parametrize("fmt", QUANT)
def test_tail_block_uses_valid_elements_only(oracle_mod, fmt):
    rng = np.random.default_rng(700 + fmt)
    for tail in (8, 16, 24):
        n = 64 + tail
        xb = to_bits(rng.standard_normal(n).astype(np.float32) * 3, F16)
        enc = oracle_mod.quantize(F16, fmt, xb)
        assert enc.size == oracle_mod.encoded_bytes(fmt, n)
        part = oracle_mod.quantize(F16, fmt, xb[64:])
        c_all, s_all, z_all = parse(enc, fmt, n)
        c_p, s_p, z_p = parse(part, fmt, tail)
        assert np.array_equal(c_all[2], c_p[0])
        assert s_all[2] == s_p[0]
        if z_all is not None:
            assert z_all[2] == z_p[0]
        assert np.all(c_all[2, tail:] == 0)  # pad codes are 0
        out = oracle_mod.dequantize(F16, fmt, enc, n)
        assert np.array_equal(out[64:], oracle_mod.dequantize(F16, fmt, part, tail))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("fmt", QUANT)
def test_roundtrip_error_bounds(oracle_mod, dtype, fmt):
    """|dequantize(quantize(x)) - x| within the format's bound per element.

    Symmetric: s/2 plus half an ulp of the output cast.  Asymmetric: s/2 +
    |m - z| + L*s*2^-11 (the fp16 rounding of the zero-point and of q*s+z)
    plus half an output ulp.  FP8: 2^-4 |x| + 2^-10 s (half a step of the
    e4m3 significand, or of its subnormal spacing) plus half an output ulp."""
    rng = np.random.default_rng(800 + fmt)
    n = 32 * 256
    xb = to_bits(rng.standard_normal(n).astype(np.float32) *
                 np.repeat(np.exp2(rng.uniform(-6, 6, n // 32)), 32).astype(np.float32), dtype)
    x = from_bits(xb, dtype).astype(np.float64)
    enc = oracle_mod.quantize(dtype, fmt, xb)
    y = from_bits(oracle_mod.dequantize(dtype, fmt, enc, n), dtype).astype(np.float64)
    _, scales, zps = parse(enc, fmt, n)
    s = np.repeat(scales.astype(np.float64), 32)
    half_ulp = np.abs(y) * (2.0 ** -11 if dtype == F16 else 2.0 ** -8) + 1e-30
    err = np.abs(y - x)
    if fmt in SYM:
        bound = s / 2 * (1 + 2.0 ** -10) + half_ulp
    elif fmt in ASYM:
        L = (1 << BITS[fmt]) - 1
        m = np.repeat(x.reshape(-1, 32).min(axis=1), 32)
        z = np.repeat(zps.astype(np.float64), 32)
        bound = s / 2 + np.abs(m - z) + L * s * 2.0 ** -11 + half_ulp + 2 * np.abs(z) * 2.0 ** -24
    else:
        bound = np.abs(x) * 2.0 ** -4 + s * 2.0 ** -10 + half_ulp
    assert np.all(err <= bound), float(np.max(err - bound))


def test_fp_format_is_passthrough(oracle_mod):
    xb = to_bits(np.random.default_rng(9).standard_normal(72).astype(np.float32), F16)
    enc = oracle_mod.quantize(F16, FP, xb)
    assert np.array_equal(enc.view(np.uint16), xb)
    assert np.array_equal(oracle_mod.dequantize(F16, FP, enc, 72), xb)


def test_zero_block_and_tiny_block(oracle_mod):
    x = np.zeros(64, np.float32)
    x[32:] = 2.0 ** -30  # a / 127 underflows fp16: scale 0, codes 0
    for fmt in QUANT:
        enc = oracle_mod.quantize(F16 if fmt != Q8A else BF16, fmt,
                                  to_bits(x, F16 if fmt != Q8A else BF16))
        codes, scales, _ = parse(enc, fmt, 64)
        assert np.all(codes == 0)
        assert scales[0] == 0
