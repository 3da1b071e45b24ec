// kvq_quant.cuh -- the plain (IEEE-division) block quantisers shared by the
// append kernels and the bit-width sweep.
//
// FP4 block ("Quantising the KV cache", section "Code"): s = RNE_e4m3(amax/6)
// saturating, a zero scale replaced by the E4M3 minimum subnormal 2^-9, codes
// RNE_e2m1(v / s) saturating, IEEE fp32 divisions, the sign of every value kept
// in its nibble.  FP8 ("Quantising the KV cache", table row "FP8 E4M3, one
// scale per tensor"): code RNE_e4m3(x / s) saturating.
#pragma once

#include "kvq_common.cuh"

namespace kvq {
namespace {

struct Block16 {
  float x[16];
  bool finite;
};

__device__ __forceinline__ Block16 load_bf16x16(const uint16_t* src) {
  Block16 b;
  const uint4 p = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  const uint32_t w[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    b.x[2 * i] = bf16_lo(w[i]);
    b.x[2 * i + 1] = bf16_hi(w[i]);
    ok &= ((w[i] & 0x7F80u) != 0x7F80u) && ((w[i] & 0x7F800000u) != 0x7F800000u);
  }
  b.finite = ok;
  return b;
}

// The E2M1 nibble of x / s: magnitude from the saturating RNE conversion of
// |x / s| (IEEE division), sign bit of x, NaN -> magnitude 7.
__device__ __forceinline__ uint32_t e2m1_pair(float x0, float x1, float s) {
  const float y0 = __fdiv_rn(x0, s);
  const float y1 = __fdiv_rn(x1, s);
  uint32_t m = e2m1x2_from_f32(fabsf(y0), fabsf(y1));
  if (isnan(y0)) m = (m & 0xF0u) | 0x7u;
  if (isnan(y1)) m = (m & 0x0Fu) | 0x70u;
  m |= (__float_as_uint(x0) >> 31) << 3;
  m |= (__float_as_uint(x1) >> 31) << 7;
  return m;
}

// Quantise one block: returns 8 packed code bytes, writes the scale byte.
__device__ __forceinline__ uint2 quantize_block(const Block16& b, uint32_t& scale_byte) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(b.x[i]));
  const float t = __fdiv_rn(amax, 6.0f);
  uint32_t sb = e4m3x2_from_f32(t, 0.0f) & 0xFFu;
  if (sb == 0u) sb = 0x01u;  // E4M3 minimum subnormal 2^-9
  const float s = e4m3_to_f32(sb);
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w0 |= e2m1_pair(b.x[2 * i], b.x[2 * i + 1], s) << (8 * i);
    w1 |= e2m1_pair(b.x[8 + 2 * i], b.x[8 + 2 * i + 1], s) << (8 * i);
  }
  scale_byte = sb;
  return make_uint2(w0, w1);
}

// E4M3 byte pair of x / s (IEEE division), sign of x, NaN -> 0x7F.
__device__ __forceinline__ uint32_t e4m3_pair(float x0, float x1, float s) {
  const float y0 = __fdiv_rn(x0, s);
  const float y1 = __fdiv_rn(x1, s);
  uint32_t m = e4m3x2_from_f32(fabsf(y0), fabsf(y1));
  m |= (__float_as_uint(x0) >> 31) << 7;
  m |= (__float_as_uint(x1) >> 31) << 15;
  if (isnan(y0)) m = (m & 0xFF00u) | 0x7Fu;
  if (isnan(y1)) m = (m & 0x00FFu) | 0x7F00u;
  return m;
}

}  // namespace
}  // namespace kvq
