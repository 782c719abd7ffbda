/*
 * Host-side proof of the division-free per-token codes of the CUDA kernels
 * (quant16_fast for int8, quant16_fp8_fast for FP8 E4M3, quant16_int4_fast
 * for int4): for every bf16 amax whose scale = amax/D (IEEE fp32 division;
 * D = 127 for int8, 448 for E4M3, 7 for int4) is at least 2^-100, and every
 * bf16 x with |x| <= amax, the corrected
 * quotient
 *     q0 = fl(x * inv), inv = fl(1/scale)
 *     rem = fma(-q0, scale, x), q1 = fma(rem, inv, q0)
 * gives the same code as the IEEE quotient fl(x / scale):
 *   int8, int4: rint(q1) (ties to even, by adding 1.5 * 2^23) equals
 *         rint(fl(x/s)) clamped to D (and never exceeds D itself); negative x
 *         follow by symmetry (every step rounds to nearest-even);
 *   E4M3: with x's sign put on q1, the nearest-even E4M3 code of q1 (all 8
 *         bits, saturated to 448) equals that of fl(x/s), for both signs of
 *         x (so -0 codes as 0x80 on both sides).
 * Prints the pair counts and the number of mismatches with and without the
 * correction step; exits 1 on any corrected mismatch.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp quant_exhaustive.c -lm
 * (contraction off so that x/scale, x*inv and the adds round on their own;
 * fmaf is the correctly rounded fused multiply-add).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_value(uint32_t bits) {
  uint32_t u = bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Nearest E4M3 code of a finite float: sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, subnormals m * 2^-9, magnitudes above 448 saturated, ties
 * to the even code. Written here from the format for this check alone. */
static unsigned e4m3_code(float v) {
  const unsigned sign = signbit(v) ? 0x80u : 0u;
  double a = fabs((double)v);
  if (a > 448.0) a = 448.0;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int ex = e2 - 1;
  if (ex < -6) ex = -6;
  const double spacing = ldexp(1.0, ex - 3);
  const double val = nearbyint(a / spacing) * spacing;
  if (val < ldexp(1.0, -6)) return sign | (unsigned)(val / ldexp(1.0, -9));
  frexp(val, &e2);
  const int vex = e2 - 1;
  return sign | (unsigned)((vex + 7) << 3) | (unsigned)((ldexp(val, -vex) - 1.0) * 8.0);
}

static float with_sign_of(float q, float x) { return copysignf(fabsf(q), x); }

int main(void) {
  const float magic = 12582912.0f; /* 1.5 * 2^23 */
  long long pairs = 0, bad = 0, bad_plain = 0, pairs8 = 0, bad8 = 0, bad8_plain = 0, pairs4 = 0, bad4 = 0,
            bad4_plain = 0;
#pragma omp parallel for schedule(dynamic, 64) \
    reduction(+ : pairs, bad, bad_plain, pairs8, bad8, bad8_plain, pairs4, bad4, bad4_plain)
  for (int a = 1; a <= 0x7F7F; ++a) { /* every positive finite bf16 amax */
    const float amax = bf16_value((uint32_t)a);
    /* int8: scale = amax / 127; int4: scale = amax / 7 */
    for (int d = 0; d < 2; ++d) {
      const float D = d == 0 ? 127.0f : 7.0f;
      volatile float s_v = amax / D;
      const float s = s_v;
      if (s < 0x1p-100f) continue;
      volatile float inv_v = 1.0f / s;
      const float inv = inv_v;
      for (uint32_t xb = 0; xb <= (uint32_t)a; ++xb) { /* every bf16 0 <= x <= amax */
        const float x = bf16_value(xb);
        volatile float qv = x / s;
        float ref = rintf(qv);
        if (ref > D) ref = D;
        volatile float q0_v = x * inv;
        const float q0 = q0_v;
        const float q1 = fmaf(fmaf(-q0, s, x), inv, q0);
        volatile float t1 = q1 + magic;
        volatile float t0 = q0 + magic;
        const float r1 = t1 - magic, r0 = t0 - magic;
        if (d == 0) {
          ++pairs;
          if (r1 != ref) ++bad;
          if (r0 != ref) ++bad_plain;
        } else {
          ++pairs4;
          if (r1 != ref) ++bad4;  /* no clamp on r1: it must not exceed 7 either */
          if (r0 != ref) ++bad4_plain;
        }
      }
    }
    /* E4M3: scale = amax / 448, both signs of x */
    volatile float s8_v = amax / 448.0f;
    const float s8 = s8_v;
    if (s8 >= 0x1p-100f) {
      volatile float inv_v = 1.0f / s8;
      const float inv = inv_v;
      for (uint32_t xb = 0; xb <= (uint32_t)a; ++xb) {
        for (int neg = 0; neg < 2; ++neg) {
          const float x = bf16_value(xb | (neg ? 0x8000u : 0u));
          volatile float qv = x / s8;
          const unsigned ref = e4m3_code(qv);
          volatile float q0_v = x * inv;
          const float q0 = q0_v;
          const float q1 = with_sign_of(fmaf(fmaf(-q0, s8, x), inv, q0), x);
          ++pairs8;
          if (e4m3_code(q1) != ref) ++bad8;
          if (e4m3_code(q0) != ref) ++bad8_plain;
        }
      }
    }
  }
  printf("pairs %lld corrected_mismatch %lld uncorrected_mismatch %lld\n", pairs, bad, bad_plain);
  printf("fp8_pairs %lld fp8_corrected_mismatch %lld fp8_uncorrected_mismatch %lld\n", pairs8, bad8, bad8_plain);
  printf("int4_pairs %lld int4_corrected_mismatch %lld int4_uncorrected_mismatch %lld\n", pairs4, bad4, bad4_plain);
  return (bad != 0 || bad8 != 0 || bad4 != 0);
}
