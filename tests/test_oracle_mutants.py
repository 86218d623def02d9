"""The pins must pin: each plausible mistake below is planted in a copy of
the oracle's C source (on the CPU), the copy is built, and at least one of
the oracle's pin tests must fail against it.  The real oracle passes all of
them (the ordinary test run)."""
import os

import numpy as np
import pytest

import oracle
import test_oracle_allreduce as TA
import test_oracle_codec as TC
import test_oracle_conversions as TV
from quantized_allreduce_codec_gb300.inputs import BF16, F16, FP, FP8, Q4, Q4A, Q6, Q8, Q8A

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "qro.c")

# (name, text in qro.c, replacement)
MUTANTS = [
    ("sym Qmax is 2^(b-1)", "static int sym_qmax(int fmt) { return (1 << (code_bits(fmt) - 1)) - 1; }",
     "static int sym_qmax(int fmt) { return (1 << (code_bits(fmt) - 1)); }"),
    ("asym levels 2^b", "static int asym_levels(int fmt) { return (1 << code_bits(fmt)) - 1; }",
     "static int asym_levels(int fmt) { return (1 << code_bits(fmt)); }"),
    ("round half away from zero", "      float r = rintf(v);\n      if (r < -qmax)", "      float r = roundf(v);\n      if (r < -qmax)"),
    ("asym rounds half away", "      float r = rintf(v); /* round half to even (default rounding mode) */",
     "      float r = roundf(v);"),
    ("no lower clamp (sym)", "      if (r < -qmax) r = -qmax;\n", ""),
    ("asym zero-point from the max", "    bc->z_bits = qro_f32_to_f16_satfinite(m);", "    bc->z_bits = qro_f32_to_f16_satfinite(M);"),
    ("asym decode subtracts z", "    return qs + z;", "    return qs - z;"),
    ("asym shift by unrounded min", "      float shifted = x[i] - bc->z;", "      float shifted = x[i] - m;"),
    ("encoder uses unrounded scale", "  float inv = 1.0f / bc->s;\n  for (int i = 0; i < cnt; ++i) {\n    float v = x[i] * inv;",
     "  float inv = qmax / a;\n  for (int i = 0; i < cnt; ++i) {\n    float v = x[i] * inv;"),
    ("scale by reciprocal multiply", "  float ratio = a / qmax;", "  float ratio = a * (1.0f / qmax);"),
    ("fp8 divisor 127", "  const float qmax = fmt == QRO_FP8 ? 448.0f : (float)sym_qmax(fmt);",
     "  const float qmax = fmt == QRO_FP8 ? 127.0f : (float)sym_qmax(fmt);"),
    ("accumulate from +0", "      for (int i = 0; i < cnt; ++i) acc[i] = (r == 0) ? xhat[i] : acc[i] + xhat[i];",
     "      for (int i = 0; i < cnt; ++i) acc[i] = (r == 0) ? 0.0f + xhat[i] : acc[i] + xhat[i];"),
    ("accumulate subtracts", "      for (int i = 0; i < cnt; ++i) acc[i] = (r == 0) ? xhat[i] : acc[i] + xhat[i];",
     "      for (int i = 0; i < cnt; ++i) acc[i] = (r == 0) ? xhat[i] : acc[i] - xhat[i];"),
    ("requantize the dtype-rounded sum", "        encode_block(fmt, acc, cnt, &bc);\n        if (wire)",
     "        for (int i = 0; i < cnt; ++i) acc[i] = widen(dtype, narrow(dtype, acc[i]));\n"
     "        encode_block(fmt, acc, cnt, &bc);\n        if (wire)"),
    ("stage 2 skipped", "    if (stages == 2) {\n      if (is_quantized(fmt)) {", "    if (stages == 3) {\n      if (is_quantized(fmt)) {"),
    ("stage 1 skips the codec", "      if (is_quantized(fmt)) {\n        block_code bc;\n        encode_block(fmt, x, cnt, &bc);\n        for (int i = 0; i < cnt; ++i) xhat[i]",
     "      if (0) {\n        block_code bc;\n        encode_block(fmt, x, cnt, &bc);\n        for (int i = 0; i < cnt; ++i) xhat[i]"),
    ("codes stored in reverse order", "  for (int i = 0; i < QRO_BLOCK; ++i) put_code(codes, b, i, bc->q[i]);",
     "  for (int i = 0; i < QRO_BLOCK; ++i) put_code(codes, b, QRO_BLOCK - 1 - i, bc->q[i]);"),
    ("no sign extension on decode", "  if (is_signed && (u >> (b - 1)) & 1u) return (int)u - (1 << b);", ""),
    ("zero-points over the scales", "    uint8_t *zp = enc + nb * cb + 2 * nb + 2 * blk;", "    uint8_t *zp = enc + nb * cb + 2 * blk;"),
    ("ties away in format rounding", "  if (frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) != 0.0)) k += 1.0;",
     "  if (frac >= 0.5) k += 1.0;"),
    ("no subnormal clamp", "  if (E < emin) E = emin;\n  int qexp", "  int qexp"),
    ("e4m3 no saturation", "  if (r > 448.0) r = 448.0;\n", ""),
    ("bf16 mantissa 6 bits", "  unsigned s = h >> 15, e = (h >> 7) & 0xFFu, m = h & 0x7Fu;",
     "  unsigned s = h >> 15, e = (h >> 7) & 0xFFu, m = h & 0x3Fu;"),
    ("fp16 saturates to inf", "    if (saturate) return (uint16_t)(sign | 0x7BFFu); /* 65504 */",
     "    if (saturate) return (uint16_t)(sign | 0x7C00u);"),
    ("tail stats over all 32", "    for (int i = 1; i < cnt; ++i) {\n      if (x[i] < m) m = x[i];",
     "    for (int i = 1; i < QRO_BLOCK; ++i) {\n      if (x[i] < m) m = x[i];"),
    ("sym absmax ignores sign", "    float ax = fabsf(x[i]);", "    float ax = x[i];"),
    ("asym lower clamp missing", "      if (r < 0.0f) r = 0.0f;\n", ""),
    ("sym and fp8 scale not saturating", "  bc->s_bits = qro_f32_to_f16_satfinite(ratio);\n  bc->s = qro_f16_to_f32(bc->s_bits);\n  if",
     "  bc->s_bits = qro_f32_to_f16(ratio);\n  bc->s = qro_f16_to_f32(bc->s_bits);\n  if"),
    ("asym scale not saturating", "    bc->s_bits = qro_f32_to_f16_satfinite(ratio);\n    bc->z_bits",
     "    bc->s_bits = qro_f32_to_f16(ratio);\n    bc->z_bits"),
    ("asym zero-point not saturating", "    bc->z_bits = qro_f32_to_f16_satfinite(m);", "    bc->z_bits = qro_f32_to_f16(m);"),
    ("more than eight ranks accepted", "  if (W < 1 || W > 8 || !valid_dtype(dtype) || !valid_format(fmt)) return -1;",
     "  if (W < 1 || W > 16 || !valid_dtype(dtype) || !valid_format(fmt)) return -1;"),
    ("cast option truncates its result to bf16",
     "    for (size_t i = 0; i < n; ++i) out[i] = qro_f32_to_bf16(qro_f16_to_f32(o16[i]));",
     "    for (size_t i = 0; i < n; ++i) {\n      float f = qro_f16_to_f32(o16[i]);\n      uint32_t u;\n"
     "      memcpy(&u, &f, 4);\n      out[i] = (uint16_t)(u >> 16);\n    }"),
    ("cast option runs the bf16 path", "  int rc = qro_allreduce(W, QRO_F16, fmt, stages, h, n, o16, wire);",
     "  int rc = qro_allreduce(W, QRO_BF16, fmt, stages, inputs, n, out, wire);\n  free(buf);\n  return rc;"),
]


def battery(o):
    """The pin tests, cheapest first, as callables on an oracle object."""
    yield lambda: TC.test_hand_worked_q8_block(o)
    yield lambda: TA.test_rejects_bad_arguments(o)
    yield lambda: TC.test_packing_known_answer_q6_q4(o)
    yield lambda: TC.test_zero_block_and_tiny_block(o)
    yield lambda: TA.test_signed_zeros_fp_path(o, F16)
    for dt in (F16, BF16):
        for st in (1, 2):
            yield lambda dt=dt, st=st: TA.test_w1_fp_identity(o, dt, st)
        for W in (2, 3):
            yield lambda dt=dt, W=W: TA.test_fp_path_is_rank_order_f32_sum(o, dt, W)
    for f in (Q8, Q6, Q4, FP8, Q8A, Q4A):
        yield lambda f=f: TC.test_tail_block_uses_valid_elements_only(o, f)
    for dt in (F16, BF16):
        for f in (Q8, Q6, Q4):
            yield lambda dt=dt, f=f: TC.test_sym_grid_roundtrip(o, dt, f)
            yield lambda dt=dt, f=f: TC.test_sym_codes_are_bruteforce_nearest(o, dt, f)
        for f in (Q8A, Q4A):
            yield lambda dt=dt, f=f: TC.test_asym_grid_roundtrip(o, dt, f)
            yield lambda dt=dt, f=f: TC.test_asym_codes_are_bruteforce_nearest(o, dt, f)
        yield lambda dt=dt: TC.test_fp8_grid_roundtrip(o, dt)
        yield lambda dt=dt: TC.test_fp8_codes_are_bruteforce_nearest(o, dt)
        for f in (FP8, Q8, Q6, Q4, Q8A, Q4A):
            yield lambda dt=dt, f=f: TA.test_w1_quantized_is_codec_roundtrip(o, dt, f)
            yield lambda dt=dt, f=f: TC.test_roundtrip_error_bounds(o, dt, f)
            for W in (2, 4):
                yield lambda dt=dt, f=f, W=W: TA.test_quantized_stages_compose_from_codec(o, dt, f, W)
    for f in (FP, FP8, Q8, Q6, Q4, Q8A, Q4A):
        for st in (1, 2):
            yield lambda f=f, st=st: TA.test_block_partition_independence(o, f, st)
    yield lambda: TV.test_e4m3_saturates(o)
    yield lambda: TV.test_f16_satfinite_is_clip_then_round(o)
    yield lambda: TV.test_bf16_decode_every_pattern(o)
    yield lambda: TV.test_f16_encode_matches_numpy(o)
    yield lambda: TV.test_bf16_encode_matches_torch(o)
    yield lambda: TV.test_e4m3_encode_matches_torch_in_range(o)
    for f in (Q8A, Q4A):
        yield lambda f=f: TA.test_asym_requantization_codes_are_bruteforce_nearest(o, f)
    for f, st in ((FP, 2), (Q4A, 2), (Q8, 1)):
        yield lambda f=f, st=st: TA.test_bf16_cast_option_is_fp16_run_between_library_casts(o, f, st)


def first_failure(o):
    for i, check in enumerate(battery(o)):
        try:
            check()
        except (AssertionError, ValueError, pytest.fail.Exception) as e:  # the last: pytest.raises saw no error
            return i, repr(e)[:120]
    return None


def test_real_oracle_passes_battery(oracle_mod):
    assert first_failure(oracle.Oracle(oracle.build())) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found exactly once: {name}"
    mutant_src = tmp_path / "qro.c"
    mutant_src.write_text(src.replace(old, new))
    so = oracle.compile_source(str(mutant_src), str(tmp_path / "libmutant.so"))
    with np.errstate(all="ignore"):
        caught = first_failure(oracle.Oracle(so))
    assert caught is not None, f"no pin caught the planted mistake: {name}"
