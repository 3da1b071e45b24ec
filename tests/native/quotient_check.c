// Exhaustive checks behind the append's division-free quotients.  Both take
// q = RN(y * r) with r = RN(1/s), then q' = fma(-fma(q, s, -y), r, q), and
// require q' == RN(y / s), the IEEE fp32 quotient:
//   1. every fp32 y in [1, 2) against every E4M3 significand s in
//      {1, 1.125, ..., 1.875} (the block scale, and the divisor 6 of amax/6);
//   2. every bf16 y in [1, 2) (the 2^7 significands of the input) against
//      every fp32 s in [1, 2) (the NVFP4 second-level scale).
// All steps scale exactly with the exponents of y and s while the values stay
// normal and the residual y - q*s is exact, so these cover every such
// dividend and divisor of each kind.
//   3. the ends of the second-level scale range the append takes this path
//      for, s in [2^-90, 2^126] (exponents -90, -89, 125, 126, every 4099th
//      significand), against every finite positive bf16 y: where the IEEE
//      quotient is finite and at least 2^-12 the two are equal; below 2^-12
//      the quotient keeps the sign and stays under 2^-11 (its E2M1 code under
//      any block scale is the signed zero); where the IEEE quotient
//      overflows the quotient is not finite either.
// Exit status 0 when every case matches.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static volatile float g_one = 1.0f;  // keeps the compiler from folding the probe below

static long check(float y, float s, float r, long* bad, const char* what) {
  const float q = y * r;
  const float q2 = fmaf(-fmaf(q, s, -y), r, q);
  const float ref = y / s;
  if (u_of(q2) != u_of(ref)) {
    if (*bad < 5) printf("%s mismatch s=%a y=%a q2=%a ref=%a\n", what, s, y, q2, ref);
    ++*bad;
  }
  return 1;
}

int main(void) {
  // fmaf must round once: (1 + 2^-23)^2 - (1 + 2^-22) is 2^-46 exactly,
  // and 0 when the product is rounded first
  const float e = g_one + 0x1p-23f;
  if (fmaf(e, e, -(g_one + 0x1p-22f)) != 0x1p-46f) {
    printf("fmaf is not fused on this host\n");
    return 2;
  }
  long bad = 0, total = 0;
  for (int m = 0; m < 8; ++m) {
    const float s = 1.0f + m / 8.0f;
    const float r = 1.0f / s;
    for (uint32_t k = 0; k < (1u << 23); ++k) total += check(f_of(0x3F800000u | k), s, r, &bad, "e4m3");
  }
  printf("e4m3 divisors: checked %ld, mismatches %ld\n", total, bad);
  const long bad1 = bad;
  total = 0;
  for (uint32_t k = 0; k < (1u << 23); ++k) {
    const float s = f_of(0x3F800000u | k);
    const float r = 1.0f / s;
    for (uint32_t j = 0; j < 128; ++j) total += check(f_of(0x3F800000u | (j << 16)), s, r, &bad, "fp32");
  }
  printf("fp32 divisors, bf16 dividends: checked %ld, mismatches %ld\n", total, bad - bad1);
  long bad3 = 0;
  total = 0;
  const int exps[4] = {-90, -89, 125, 126};
  for (int ei = 0; ei < 4; ++ei)
    for (uint32_t k = 0; k < (1u << 23); k += 4099) {
      const float s = ldexpf(f_of(0x3F800000u | k), exps[ei]);
      const float r = 1.0f / s;
      for (uint32_t xb = 1; xb < 0x7F80u; ++xb) {
        const float y = f_of(xb << 16);
        const float q = y * r;
        const float q2 = fmaf(-fmaf(q, s, -y), r, q);
        const float ref = y / s;
        int ok;
        if (isinf(ref)) ok = !isfinite(q2);
        else if (ref >= 0x1p-12f) ok = u_of(q2) == u_of(ref);
        else ok = !signbit(q2) && q2 < 0x1p-11f;
        ++total;
        if (!ok) {
          if (bad3 < 5) printf("range mismatch s=%a y=%a q2=%a ref=%a\n", s, y, q2, ref);
          ++bad3;
        }
      }
    }
  printf("second-level scale range ends: checked %ld, mismatches %ld\n", total, bad3);
  return bad != 0 || bad3 != 0;
}
