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
//   4. the FP4 codes with an approximate reciprocal: for every positive
//      finite E4M3 block scale s (normal and subnormal), every r within two
//      ulps of RN(1/s) and every finite bf16 x the block could hold (|x| at
//      most 8 s, any x when s is the saturated 448), the saturating round-to-
//      nearest-even E2M1 code (sign kept) of the corrected quotient
//      fma(-fma(q, s, -x), r, q), q = x * r, equals the code of x / s.  (The
//      value itself may differ from x / s by an ulp; on an E2M1 midpoint it
//      does not, and off one it stays on the same side.)
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

// E2M1 code of v: sign bit 8, magnitude code by the grid's midpoints, ties to
// the even code, saturating above 6.
static int e2m1_code(float v) {
  static const float mid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  const float a = fabsf(v);
  int c = 0;
  for (int i = 0; i < 7; ++i) {
    if (a > mid[i]) {
      c = i + 1;
    } else {
      if (a == mid[i]) c = (i % 2 == 0) ? i : i + 1;
      break;
    }
  }
  return (signbit(v) ? 8 : 0) | c;
}

static float e4m3_value(int b) {  // b in 1..0x7E (positive finite)
  const int e = b >> 3, m = b & 7;
  return e ? ldexpf(1.0f + m / 8.0f, e - 7) : ldexpf((float)m, -9);
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
  long bad4 = 0;
  total = 0;
  for (int b = 1; b <= 0x7E; ++b) {
    const float s = e4m3_value(b);
    const uint32_t r0 = u_of(1.0f / s);
    for (int k = -2; k <= 2; ++k) {
      const float r = f_of(r0 + (uint32_t)k);
      for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
        if ((xb & 0x7F80u) == 0x7F80u) continue;  // Inf and NaN take the IEEE path
        const float x = f_of(xb << 16);
        // reachable pairs only: a block's scale s = RNE_e4m3(amax / 6) is at
        // least amax / 6.4 unless it saturated at 448, so |x| <= 6.4 s
        if (b != 0x7E && !(fabsf(x) <= 8.0f * s)) continue;
        const float q = x * r;
        const float q2 = fmaf(-fmaf(q, s, -x), r, q);
        ++total;
        if (e2m1_code(q2) != e2m1_code(x / s)) {
          if (bad4 < 5) printf("code mismatch s=%a r=%a x=%a q2=%a ref=%a\n", s, r, x, q2, x / s);
          ++bad4;
        }
      }
    }
  }
  printf("approximate reciprocals, e2m1 codes: checked %ld, mismatches %ld\n", total, bad4);
  return bad != 0 || bad3 != 0 || bad4 != 0;
}
