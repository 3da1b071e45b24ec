// Exhaustive check behind the NVFP4 append's division-free quotient: for every
// fp32 y in [1, 2) and every E4M3 significand s in {1, 1.125, ..., 1.875},
// q' = fma(-fma(q, s, -y), r, q) with r = RN(1/s) and q = RN(y * r) equals the
// IEEE fp32 quotient RN(y / s).  All steps scale exactly with the exponents of y
// and s while the values stay normal, so this covers every y and every E4M3
// scale (subnormal E4M3 scales have significands in the same set).  Exit status
// 0 when every case matches.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
int main(void) {
  long bad = 0, total = 0;
  for (int m = 0; m < 8; ++m) {
    const float s = 1.0f + m / 8.0f;
    const float r = 1.0f / s;
    for (uint32_t k = 0; k < (1u << 23); ++k) {
      const float y = f_of(0x3F800000u | k);
      const float q = y * r;
      const float q2 = fmaf(-fmaf(q, s, -y), r, q);
      const float ref = y / s;
      ++total;
      if (u_of(q2) != u_of(ref)) {
        if (bad < 5) printf("mismatch s=%g y=%a q2=%a ref=%a\n", s, y, q2, ref);
        ++bad;
      }
    }
  }
  printf("checked %ld, mismatches %ld\n", total, bad);
  return bad != 0;
}
