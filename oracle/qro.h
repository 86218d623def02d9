/*
 * qro.h -- CPU oracle for the quick-allreduce block codec and the emulated
 * one- and two-stage allreduce.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, deliberately unoptimised
 * restatement of what the data path computes, used to check the CUDA library
 * bit for bit.  Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg may call it.  It shares no code, header or table with the
 * CUDA library, and it includes nothing from it.
 *
 * Sources (web pages):
 *   [P1] vLLM PR #18473, "Integrate quick allreduce and select the best
 *        allreduce implementation": the formats 1stage f16 and 2stage
 *        f16/fp8/Q8/Q6/Q4 (opening description; tp2 kernel timing table).
 *   [P2] vLLM PR #16804, "Add quickreduce as alternative to custom allreduce":
 *        int4/int8 symmetric and asymmetric quantization (opening
 *        description); one shot for small buffers, two shot for larger ones
 *        (review discussion).
 *   [P4] vLLM API docs, "vllm.distributed.device_communicators.
 *        quick_all_reduce": QuickReduceRegime (FP=0, INT8=1, INT6=2, INT4=3),
 *        supported dtypes fp16/bf16, byte size a multiple of 16,
 *        out-of-place quick_all_reduce.
 * The pages give no block layout, scale type, rounding or packing.  The
 * readings used here (32-element blocks, an fp16 scale per block, an fp16
 * zero-point for the asymmetric formats, round-half-to-even, saturating
 * codes, little-endian Q6/Q4 packing, a structure-of-arrays encoded buffer)
 * are stated at each function in qro.c.
 */
#ifndef QRO_H
#define QRO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Enum values repeated here on purpose (the oracle includes nothing from the
 * library); a test checks that both sides agree.  0..3 follow
 * QuickReduceRegime on [P4]; 4..6 are the fp8 format of [P1] and the
 * asymmetric formats of [P2]. */
enum { QRO_F16 = 0, QRO_BF16 = 1, QRO_BF16_AS_F16 = 2 };
enum {
  QRO_FP = 0, QRO_Q8 = 1, QRO_Q6 = 2, QRO_Q4 = 3,
  QRO_FP8 = 4, QRO_Q8A = 5, QRO_Q4A = 6
};
#define QRO_BLOCK 32

/* Scalar conversions (exported so the tests can pin them to library casts). */
float    qro_f16_to_f32(uint16_t h);
uint16_t qro_f32_to_f16(float v);          /* RNE, overflow -> inf          */
uint16_t qro_f32_to_f16_satfinite(float v);/* RNE, overflow -> +-65504      */
float    qro_bf16_to_f32(uint16_t h);
uint16_t qro_f32_to_bf16(float v);         /* RNE, overflow -> inf          */
float    qro_e4m3_to_f32(uint8_t c);
uint8_t  qro_f32_to_e4m3_satfinite(float v); /* RNE, overflow -> +-448      */

/* Bytes of one encoded message of n elements (codes, then scales, then
 * zero-points); FP passthrough is n*2.  0 for an unknown format. */
size_t qro_encoded_bytes(int fmt, size_t n);

/* Encode / decode one message.  in/out hold n 16-bit values of dtype.
 * Return 0 on success, -1 on a bad argument. */
int qro_quantize(int dtype, int fmt, const uint16_t *in, size_t n, uint8_t *enc);
int qro_dequantize(int dtype, int fmt, const uint8_t *enc, size_t n, uint16_t *out);

/* Emulated allreduce of W messages of n elements each (out-of-place).
 * wire (may be NULL) receives the stage-2 payload for stages == 2.
 * dtype QRO_BF16_AS_F16: bf16 messages are rounded to fp16 first, the fp16
 * allreduce runs, and its result is rounded back to bf16 (the bf16 -> fp16
 * cast option of init_quick_all_reduce on the vLLM quick_all_reduce page);
 * the payload is the fp16 run's. */
int qro_allreduce(int W, int dtype, int fmt, int stages,
                  const uint16_t *const *inputs, size_t n,
                  uint16_t *out, uint8_t *wire);

#ifdef __cplusplus
}
#endif
#endif
