"""The integer identities the kernels' code packing and unpacking rest on,
checked on the CPU with the constants the device code uses (no GPU).

Packing: a rounding sum t = RN(v + 1.5*2^23) holding the integer code q reads,
as a 32-bit pattern, 0x4B400000 + q.  So a weighted sum of eight such patterns
minus the magic pattern's share leaves the biased codes in their fields with
no carries, and one XOR turns biased symmetric codes into two's-complement
fields.  Unpacking: a field masked in place under the exponent that makes its
lowest bit the units place reads, as binary32, 2^e + field."""
import struct

import numpy as np

M = 0x4B400000  # binary32 pattern of 1.5 * 2^23
U32 = 0xFFFFFFFF


def pattern(q: int) -> int:
    return struct.unpack("<I", struct.pack("<f", 12582912.0 + q))[0]


def pack4(qs, sym):
    """The device's 4-bit packing of eight codes (pack_codes)."""
    t = [pattern(q) for q in qs]
    fix = ((8 if sym else 0) - M) * 0x11111111 & U32
    p01, p23 = (t[1] * 16 + t[0]) & U32, (t[3] * 16 + t[2]) & U32
    p45, p67 = (t[5] * 16 + t[4]) & U32, (t[7] * 16 + t[6]) & U32
    acc = ((p67 * 256 + p45) * 65536 + (p23 * 256 + p01) + fix) & U32
    return acc ^ 0x88888888 if sym else acc


def pack6(qs):
    """The device's 6-bit packing of eight symmetric codes: (word 0, low 16 bits of word 1)."""
    t = [pattern(q) for q in qs]
    off = (M - 32) & U32
    w0 = 1 + (1 << 6) + (1 << 12) + (1 << 18) + (1 << 24) + (1 << 30)
    lo = ((t[1] * 64 + t[0]) + (t[3] * 64 + t[2]) * 4096 + (t[5] * 64 + t[4]) * 16777216) & U32
    hi = ((t[5] >> 2) + t[6] * 16 + t[7] * 1024 - ((off >> 2) + off * 16 + off * 1024)) & U32
    return ((lo - off * w0) & U32) ^ 0x20820820, (hi ^ 0x8208) & 0xFFFF


def fields(qs, bits):
    v = 0
    for j, q in enumerate(qs):
        v |= (q & ((1 << bits) - 1)) << (bits * j)
    return v


def test_rounding_sum_pattern_is_magic_plus_code():
    for q in range(-300, 301):
        assert pattern(q) == (M + q) & U32


def test_4bit_packing_symmetric_and_asymmetric():
    rng = np.random.default_rng(1)
    for pos in range(8):  # every code value at every position, the others at the range ends
        for q in range(-7, 8):
            for fill in (-7, 7, 0):
                qs = [fill] * 8
                qs[pos] = q
                assert pack4(qs, True) == fields(qs, 4)
        for q in range(16):
            for fill in (0, 15):
                qs = [fill] * 8
                qs[pos] = q
                assert pack4(qs, False) == fields(qs, 4)
    for _ in range(20000):
        qs = rng.integers(-7, 8, 8).tolist()
        assert pack4(qs, True) == fields(qs, 4)
        qa = rng.integers(0, 16, 8).tolist()
        assert pack4(qa, False) == fields(qa, 4)


def test_6bit_packing():
    rng = np.random.default_rng(2)
    for pos in range(8):
        for q in range(-31, 32):
            for fill in (-31, 31, 0):
                qs = [fill] * 8
                qs[pos] = q
                s = fields(qs, 6)
                assert pack6(qs) == (s & U32, (s >> 32) & 0xFFFF)
    for _ in range(20000):
        qs = rng.integers(-31, 32, 8).tolist()
        s = fields(qs, 6)
        assert pack6(qs) == (s & U32, (s >> 32) & 0xFFFF)


def pow2_bits(e: int) -> int:
    return (127 + e) << 23


def as_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits & U32))[0]


def test_4bit_unpacking_by_exponent():
    # nibble k of a word, at bit 4k (after a 16-bit shift for k >= 4), masked
    # in place under 2^(23-4k'): value 2^(23-4k') + nibble; symmetric codes get
    # bit 3 flipped (biased by 8)
    for sym in (True, False):
        f = 8 if sym else 0
        for kp in range(4):
            p = 4 * kp
            for c in range(16):  # the stored nibble
                w = c << p
                val = as_float((w & (0xF << p)) ^ (pow2_bits(23 - p) | (f << p)))
                q = val - (2.0 ** (23 - p) + f)
                want = (c ^ 8) - 8 if sym else c  # two's complement (sym) or unsigned code
                assert q == want, (sym, kp, c, q)


def test_6bit_unpacking_by_exponent():
    # a 6-bit field at bit p <= 17, masked in place under 2^(23-p), sign bit
    # flipped: 2^(23-p) + field + 32
    for p in (0, 6, 12, 4, 10):
        for c in range(64):
            w = c << p
            val = as_float((w & (0x3F << p)) ^ (pow2_bits(23 - p) | (0x20 << p)))
            q = val - (2.0 ** (23 - p) + 32)
            assert q == (c ^ 32) - 32, (p, c, q)
