/* Exhaustive check of the write kernel's division method against IEEE
 * binary32 division.
 *
 * The kernel divides a bf16 value x by a per-head scale s with a
 * precomputed reciprocal r = RN(1/s) and one residual correction (the
 * Markstein iteration): q0 = RN(x * r); e = RN(q0 * -s + x) (fused);
 * q = RN(e * r + q0) (fused).  Rounding depends only on the
 * significands of x and s while the quotient stays normal, so checking every
 * bf16 significand (128) against every binary32 significand (2^23), with
 * both in [1, 2), covers every normal quotient.  Prints the number of
 * mismatches (0 expected). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bits_to_f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

int main(void) {
  long long bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int64_t ms = 0; ms < (1 << 23); ++ms) {
    const float s = bits_to_f(0x3F800000u | (uint32_t)ms);       /* [1, 2) */
    const float r = 1.0f / s;                                      /* RN(1/s) */
    for (uint32_t mx = 0; mx < 128; ++mx) {
      const float x = bits_to_f(0x3F800000u | (mx << 16));        /* bf16 in [1, 2) */
      const float want = x / s;
      const float q0 = x * r;
      const float e = fmaf(q0, -s, x);
      const float q = fmaf(e, r, q0);
      if (q != want) bad += 1;
    }
  }
  printf("%lld\n", bad);
  return 0;
}
