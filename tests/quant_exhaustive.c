/*
 * Host-side proof of the int8 code's division-free path (the CUDA kernels'
 * quant16_fast): for every bf16 amax whose scale = amax/127 (IEEE fp32
 * division) is at least 2^-100, and every bf16 x with |x| <= amax, the
 * corrected quotient
 *     q0 = fl(x * inv), inv = fl(1/scale)
 *     rem = fma(-q0, scale, x), q1 = fma(rem, inv, q0)
 * rounds (ties to even, here by adding 1.5 * 2^23) to the same integer as the
 * IEEE quotient fl(x / scale) does. Negative x follow by symmetry (every step
 * rounds to nearest-even, which is symmetric). Prints the pair count and the
 * number of mismatches of the corrected and of the uncorrected quotient;
 * exits 1 on any corrected mismatch.
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

int main(void) {
  long long pairs = 0, bad = 0, bad_plain = 0;
  const float magic = 12582912.0f; /* 1.5 * 2^23 */
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, bad, bad_plain)
  for (int a = 1; a <= 0x7F7F; ++a) { /* every positive finite bf16 amax */
    const float amax = bf16_value((uint32_t)a);
    volatile float s_v = amax / 127.0f;
    const float s = s_v;
    if (s < 0x1p-100f) continue; /* those rows take the IEEE division path */
    volatile float inv_v = 1.0f / s;
    const float inv = inv_v;
    for (uint32_t xb = 0; xb <= (uint32_t)a; ++xb) { /* every bf16 0 <= x <= amax */
      const float x = bf16_value(xb);
      volatile float qv = x / s;
      float ref = rintf(qv);
      if (ref > 127.0f) ref = 127.0f;
      volatile float q0_v = x * inv;
      const float q0 = q0_v;
      const float rem = fmaf(-q0, s, x);
      const float q1 = fmaf(rem, inv, q0);
      volatile float t1 = q1 + magic;
      volatile float t0 = q0 + magic;
      const float fast = t1 - magic, plain = t0 - magic;
      ++pairs;
      if (fast != ref) ++bad;
      if (plain != ref) ++bad_plain;
    }
  }
  printf("pairs %lld corrected_mismatch %lld uncorrected_mismatch %lld\n", pairs, bad, bad_plain);
  return bad != 0;
}
