/*
 * Checks the scale division used by the CUDA kernels against IEEE division.
 *
 * The kernels compute a / L (L = 127, 31, 7, 448, 255, 15: the largest code
 * magnitude or level count of each format) without a divide instruction:
 *   y  = RN(1 / L)                 (a compile-time constant)
 *   q0 = RN(a * y)
 *   r  = fma(-q0, L, a)            (the exact remainder)
 *   q1 = fma(r, y, q0)
 * (one remainder correction after a correctly rounded reciprocal, the method
 * of P. Markstein, "Computation of elementary functions on the IBM RISC
 * System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  The scale that is
 * stored is h(q1), h = round to fp16 (nearest even, saturating).  This
 * program checks h(q1) == h(a / L) for every non-negative finite binary32 a
 * (mode "all"), or for every a whose low `stride_log2` mantissa bits are a
 * fixed pattern (sampled mode), and also counts where q1 != a / L itself.
 *
 * Usage: scale_division_check [stride_log2]   (0 = every value)
 * Prints one line per L: "L=<L> checked=<n> quotient_mismatch=<m>
 * scale_mismatch=<k> max_mismatch_quotient=<v>"; exits 1 if any scale differs.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* fp16 rounding of a non-negative value, nearest even, saturating: returns
 * the rounded value as a double (only equality of results matters here). */
static double h(float v) {
  double a = v;
  if (a == 0.0) return 0.0;
  int E;
  frexp(a, &E);
  E -= 1;
  if (E < -14) E = -14;
  double q = ldexp(a, -(E - 10));
  double k = floor(q), fr = q - k;
  if (fr > 0.5 || (fr == 0.5 && fmod(k, 2.0) != 0.0)) k += 1.0;
  double r = ldexp(k, E - 10);
  return r > 65504.0 ? 65504.0 : r;
}

int main(int argc, char **argv) {
  int stride_log2 = argc > 1 ? atoi(argv[1]) : 0;
  const float Ls[] = {127.f, 31.f, 7.f, 448.f, 255.f, 15.f};
  int failed = 0;
  for (int i = 0; i < 6; ++i) {
    const float L = Ls[i];
    const float y = 1.0f / L;
    unsigned long long n = 0, qbad = 0, sbad = 0;
    float worst = 0.0f;
    const uint32_t step = 1u << stride_log2;
    /* every exponent; within it every `step`-th mantissa, plus the last one */
    for (uint32_t u = 0; u < 0x7F800000u; u += step) {
      for (int edge = 0; edge < (step > 1 ? 2 : 1); ++edge) {
        const uint32_t w = edge ? (u | (step - 1)) : u;
        const float a = from_bits(w);
        const float q0 = a * y;
        const float r = fmaf(-q0, L, a);
        const float q1 = fmaf(r, y, q0);
        const float ref = a / L;
        ++n;
        if (q1 != ref) {
          ++qbad;
          if (ref > worst) worst = ref;
          if (h(q1) != h(ref)) ++sbad;
        }
      }
    }
    printf("L=%g checked=%llu quotient_mismatch=%llu scale_mismatch=%llu max_mismatch_quotient=%g\n",
           L, n, qbad, sbad, worst);
    if (sbad) failed = 1;
  }
  return failed;
}
