"""Pins for the oracle's scalar format conversions.

Each conversion is written in the oracle from the format's definition (sign,
biased exponent, significand).  Here it is checked against independent
library casts: numpy's float16 (IEEE binary16, round-half-to-even), torch's
CPU bfloat16 and float8_e4m3fn (OCP e4m3fn) casts, exhaustively over every
bit pattern for decoding and over random values plus every exact tie for
encoding.
"""
import numpy as np
import pytest
import torch


def _all_u16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _same_f32(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.all(both_nan | (a.view(np.uint32) == b.view(np.uint32)))


def test_f16_decode_every_pattern(oracle_mod):
    bits = _all_u16()
    ref = bits.view(np.float16).astype(np.float32)
    assert _same_f32(oracle_mod.f16_to_f32(bits), ref)


def test_bf16_decode_every_pattern(oracle_mod):
    bits = _all_u16()
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert _same_f32(oracle_mod.bf16_to_f32(bits), ref)


def test_e4m3_decode_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert _same_f32(oracle_mod.e4m3_to_f32(codes), ref)


def _f16_ties():
    """Every exact midpoint between adjacent finite fp16 values (both signs)."""
    b = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = b.view(np.float16).astype(np.float64)
    hi = (b + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)  # 12 significant bits: exact in binary32
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)
    return np.concatenate([mid, -mid])


def _random_f32(rng, count, lo_exp, hi_exp):
    mant = rng.random(count) + 1.0
    exps = rng.integers(lo_exp, hi_exp, count)
    sign = np.where(rng.random(count) < 0.5, -1.0, 1.0)
    return (sign * np.ldexp(mant, exps)).astype(np.float32)


def test_f16_encode_matches_numpy(oracle_mod):
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        _random_f32(rng, 20000, -30, 17),          # subnormal .. overflow range
        _f16_ties(),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0**-25,
                  2.0**-25 * 1.0000001, 3 * 2.0**-26, np.inf, -np.inf], np.float32),
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = oracle_mod.f32_to_f16(vals)
    assert np.array_equal(got, ref)


def test_f16_satfinite_is_clip_then_round(oracle_mod):
    rng = np.random.default_rng(12)
    vals = np.concatenate([_random_f32(rng, 5000, -30, 20),
                           np.array([65504.0, 65519.0, 65520.0, 1e30, -1e30, np.inf, -np.inf],
                                    np.float32)])
    ref = np.clip(vals, -65504.0, 65504.0).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle_mod.f32_to_f16_satfinite(vals), ref)


def test_bf16_encode_matches_torch(oracle_mod):
    rng = np.random.default_rng(13)
    b = rng.integers(0, 0x7F7F, 20000).astype(np.uint16)
    lo = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    hi = torch.from_numpy((b + 1).view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    ties = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([_random_f32(rng, 20000, -140, 128), ties, -ties,
                           np.array([0.0, -0.0, 3.3895e38, np.inf, -np.inf], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.f32_to_bf16(vals), ref)


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(14)
    codes = np.arange(0, 0x7E, dtype=np.uint8)  # finite non-negative codes below 448
    lo = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    hi = torch.from_numpy((codes + 1).copy()).view(torch.float8_e4m3fn).double().numpy()
    ties = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([_random_f32(rng, 20000, -14, 9), ties, -ties,
                           np.array([0.0, -0.0, 448.0, -448.0, 464.0, -464.0, 2.0**-10,
                                     2.0**-11, -2.0**-11], np.float32)])
    vals = vals[np.abs(vals) <= 464.0]  # torch turns larger magnitudes into NaN
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.f32_to_e4m3_satfinite(vals), ref)


def test_e4m3_saturates(oracle_mod):
    vals = np.array([465.0, 480.0, 1e6, np.inf, -465.0, -1e6, -np.inf], np.float32)
    got = oracle_mod.f32_to_e4m3_satfinite(vals)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE]


@pytest.mark.parametrize("pattern", [0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001])
def test_f16_roundtrip_through_f32(oracle_mod, pattern):
    v = oracle_mod.f16_to_f32([pattern])
    assert oracle_mod.f32_to_f16(v)[0] == pattern
