// kvq_append.cuh -- the FP4/NVFP4 quantise-and-store of one append work item,
// shared by the append kernel (kvq_append.cu) and the decode kernel's fused
// append of each sequence's newest token (kvq_decode.cu).
//
// FP4 block quantiser ("Quantising the KV cache", section "Code"): for each
// 16-channel block of one token and one kv head, s = RNE_e4m3(amax / 6)
// saturating (a zero scale becomes the E4M3 min subnormal 2^-9), then each
// value becomes RNE_e2m1(v / s) saturating, with both divisions IEEE fp32 and
// the sign of every value kept in its nibble.  Finite blocks take a
// division-free path whose codes equal those of the IEEE divisions
// (reciprocal quotient plus one exact residual correction, argued at
// block_quotient; for the codes the reciprocal of the block scale may be the
// hardware's approximate one, argued at scale_recip); blocks holding Inf or
// NaN take the plain IEEE-division quantiser.
#pragma once

#include "kvq_common.cuh"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

// x / s for a finite bf16 value x and an E4M3 scale s, accurate enough that
// the saturating RNE conversion to E2M1 gives the code of the exact quotient
// (and so of the IEEE fp32 division).  q = x * RN(1/s), then one residual
// step q - (q*s - x) * RN(1/s) (Markstein's correction of a reciprocal
// quotient).  Why this suffices: x has 8 significant bits and every E2M1
// rounding midpoint tau * s at most 7, so a quotient that is not on a
// midpoint sits at least 2^-9 (relative) away from one, far beyond the
// error of q; on a midpoint x = tau * s the residual q*s - x is exact (a
// one-ulp step of q times s) and the corrected value rounds to tau itself.
// The residual is taken as q*s - x so that x = -0.0 gives -0.0 (the sign of
// every value is kept in its nibble).
__device__ __forceinline__ float block_quotient(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  return __fmaf_rn(-__fmaf_rn(q, s, -x), r, q);
}

// The reciprocal of a block scale for block_quotient on bf16 values: the
// hardware's approximate reciprocal.  The E2M1 code of the corrected quotient
// is that of x / s for any r within two ulps of RN(1/s) (checked on the host
// for every E4M3 scale, every such r and every bf16 value the block can
// hold); on a midpoint x = tau * s the residual stays exact and the
// correction lands on tau, off one the quotient stays on its side.  s is a
// normal fp32 value in [2^-9, 448], so the flush-to-zero form is exact.
__device__ __forceinline__ float scale_recip(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(s));
  return r;
}

// Four pairs of fp32 values to four E2M1 byte pairs (saturating RNE, sign
// kept): byte i = code(a[2i]) | code(a[2i+1]) << 4.
__device__ __forceinline__ uint32_t e2m1x8_from_f32(float a0, float a1, float a2, float a3, float a4, float a5,
                                                    float a6, float a7) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// Scale byte of a block from its amax: RNE_e4m3(amax / 6) saturating, 0 -> 2^-9.
// amax / 6 by the same corrected reciprocal quotient: every E4M3 rounding
// midpoint has at most 5 significant bits, so 6 * midpoint has at most 7 and
// the argument above carries over (a bf16 amax on a midpoint is exact, any
// other sits 2^-9 away).
__device__ __forceinline__ uint32_t block_scale_byte(float amax) {
  constexpr float kSixth = 1.0f / 6.0f;  // RN(1/6)
  const uint32_t sb = e4m3x2_from_f32(block_quotient(amax, 6.0f, kSixth), 0.0f) & 0xFFu;
  return sb == 0u ? 0x01u : sb;
}

// Largest magnitude of 16 bf16 values (packed max of absolute values that
// propagates NaN): bf16 bits, >= 0x7F80 when the block holds Inf or NaN.
__device__ __forceinline__ uint32_t bmax_abs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t block_amax_bits(const uint32_t (&w)[8]) {
  const uint32_t m = bmax_abs(bmax_abs(bmax_abs(w[0], w[1]), bmax_abs(w[2], w[3])),
                              bmax_abs(bmax_abs(w[4], w[5]), bmax_abs(w[6], w[7])));
  return bmax_abs(m, __byte_perm(m, 0u, 0x1032u)) & 0x7FFFu;
}

// K: 8 code bytes of one finite block (channel 2i low nibble of byte i).
__device__ __forceinline__ uint2 k_codes_finite(const uint32_t (&w)[8], float s, float r) {
  uint32_t out[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t* u = w + 4 * half;
    out[half] = e2m1x8_from_f32(
        block_quotient(bf16_lo(u[0]), s, r), block_quotient(bf16_hi(u[0]), s, r),
        block_quotient(bf16_lo(u[1]), s, r), block_quotient(bf16_hi(u[1]), s, r),
        block_quotient(bf16_lo(u[2]), s, r), block_quotient(bf16_hi(u[2]), s, r),
        block_quotient(bf16_lo(u[3]), s, r), block_quotient(bf16_hi(u[3]), s, r));
  }
  return make_uint2(out[0], out[1]);
}

// One token-pair V item: byte c holds channel c of tokens 2i (low nibble) and
// 2i+1 (high nibble).  An absent token (not new in this call) is passed as
// zeros and contributes zero nibbles; the caller keeps the old ones.
__device__ __forceinline__ uint4 v_pair_codes_finite(const uint32_t (&w0)[8], float s0, float r0,
                                                     const uint32_t (&w1)[8], float s1, float r1) {
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t a = w0[2 * q], b = w0[2 * q + 1], c = w1[2 * q], d = w1[2 * q + 1];
    out[q] = e2m1x8_from_f32(
        block_quotient(bf16_lo(a), s0, r0), block_quotient(bf16_lo(c), s1, r1),
        block_quotient(bf16_hi(a), s0, r0), block_quotient(bf16_hi(c), s1, r1),
        block_quotient(bf16_lo(b), s0, r0), block_quotient(bf16_lo(d), s1, r1),
        block_quotient(bf16_hi(b), s0, r0), block_quotient(bf16_hi(d), s1, r1));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

struct Raw16 {
  uint32_t w[8];
  float amax;
  bool finite;
};

__device__ __forceinline__ void load_raw16(const uint16_t* src, Raw16& b) {
  const uint4 p = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  b.w[0] = p.x; b.w[1] = p.y; b.w[2] = p.z; b.w[3] = p.w;
  b.w[4] = q.x; b.w[5] = q.y; b.w[6] = q.z; b.w[7] = q.w;
  const uint32_t a = block_amax_bits(b.w);
  b.amax = __uint_as_float(a << 16);
  b.finite = a < 0x7F80u;
}

// Spread 8 nibbles (nibble c at bits 4c) to 8 bytes (nibble c in the low half
// of byte c).
__device__ __forceinline__ uint64_t spread_nibbles(uint32_t w) {
  uint64_t x = w;
  x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
  x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
  x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
  return x;
}

// The plain IEEE-division quantiser on x / S (S = 1: the block itself, an
// exact division), for blocks holding Inf or NaN and for NVFP4 caches.
// Returns the 8 code bytes, the scale byte and whether a value was not finite.
__device__ __noinline__ uint4 quantize_plain(const uint16_t* src, float S) {
  Block16 blk = load_bf16x16(src);
  bool ok = blk.finite;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    blk.x[i] = __fdiv_rn(blk.x[i], S);
    ok &= isfinite(blk.x[i]);
  }
  blk.finite = ok;
  uint32_t sb;
  const uint2 q = quantize_block(blk, sb);
  return make_uint4(q.x, q.y, sb, ok ? 0u : 1u);
}

// NVFP4 block: the FP4 quantiser on y = x / S, S the kv head's fp32
// second-level scale, with the codes and scale byte of the IEEE fp32
// divisions and no division on the way:
//   y = block_quotient(x, S, RN(1/S)) is the IEEE fp32 x / S for every bf16
//     x and every fp32 S while the residual x - q*S is exact: checked
//     exhaustively over the 2^7 significands of x against all 2^23
//     significands of S, the steps scaling exactly with both exponents.  The
//     residual is a multiple of about 2^-47 |x|, exact down to |x| = 2^-102;
//     with S >= 2^-90 a smaller x gives |x / S| < 2^-12, far under the first
//     E2M1 midpoint of any block scale (s >= 2^-9), where only the sign
//     reaches the code, and the sign is always kept.  S < 2^-90 (where tiny
//     x would give wrong codes) and S > 2^126 (a subnormal 1/S) take the
//     IEEE path;
//   max |y| = RN(max |x| / S) (rounding is monotone), taken once per block;
//   amax(y) / 6 and y / s by block_quotient as well: 6 and every E4M3 scale
//     have E4M3 significands, for which that quotient equals the IEEE one
//     for every fp32 dividend (exhaustive over the 2^23 significands).
// nv_fast_scale says whether S is in [2^-90, 2^126]; a block whose largest
// quotient is not finite (Inf/NaN input or overflow of x / S) returns false
// and takes quantize_plain, which flags it.
__device__ __forceinline__ bool nv_fast_scale(float S) { return S >= 0x1p-90f && S <= 0x1p126f; }

__device__ __forceinline__ bool nv_quotients(const Raw16& b, float S, float R, float (&y)[16], uint32_t& sb) {
  if (!b.finite) return false;
  const float ya = block_quotient(b.amax, S, R);
  if (!(ya <= 3.40282347e38f)) return false;
  sb = block_scale_byte(ya);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y[2 * i] = block_quotient(bf16_lo(b.w[i]), S, R);
    y[2 * i + 1] = block_quotient(bf16_hi(b.w[i]), S, R);
  }
  return true;
}

// 8 code bytes of 16 quotients (channel 2i in the low nibble of byte i).
__device__ __forceinline__ uint2 k_codes_f32(const float (&y)[16], float s, float r) {
  uint32_t out[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float* a = y + 8 * half;
    out[half] = e2m1x8_from_f32(block_quotient(a[0], s, r), block_quotient(a[1], s, r), block_quotient(a[2], s, r),
                                block_quotient(a[3], s, r), block_quotient(a[4], s, r), block_quotient(a[5], s, r),
                                block_quotient(a[6], s, r), block_quotient(a[7], s, r));
  }
  return make_uint2(out[0], out[1]);
}

// Token-pair V codes of two tokens' quotients: byte c holds channel c of
// token 0 (low nibble) and token 1 (high nibble).
__device__ __forceinline__ uint4 v_pair_codes_f32(const float (&y0)[16], float s0, float r0, const float (&y1)[16],
                                                  float s1, float r1) {
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = 4 * q;
    out[q] = e2m1x8_from_f32(block_quotient(y0[c], s0, r0), block_quotient(y1[c], s1, r1),
                             block_quotient(y0[c + 1], s0, r0), block_quotient(y1[c + 1], s1, r1),
                             block_quotient(y0[c + 2], s0, r0), block_quotient(y1[c + 2], s1, r1),
                             block_quotient(y0[c + 3], s0, r0), block_quotient(y1[c + 3], s1, r1));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// 16-channel blocks per K item (one token) and per V item (one token pair).
constexpr int kAppendBlocksK = 2;
constexpr int kAppendBlocksV = 1;

// Pool group holding position `pos` of sequence b, kv head h (its slot in the
// group in `ls`), or nullptr after setting PAGE_OOB.
template <int D>
__device__ __forceinline__ uint8_t* fp4_group(const kvq_cache& c, int b, int64_t pos, int h, int& ls, int32_t* flag) {
  const int lg_p = __ffs(c.page_size) - 1;
  const int lg_g = lg_p < 7 ? lg_p : 7;
  const int G = 1 << lg_g;
  const int64_t pg = pos >> lg_p;
  const int slot = (int)(pos & (c.page_size - 1));
  if (pg >= c.max_pages_per_seq) {
    set_flag(flag, KVQ_FLAG_PAGE_OOB);
    return nullptr;
  }
  const int64_t phys = c.page_table ? (int64_t)__ldg(c.page_table + (int64_t)b * c.max_pages_per_seq + pg)
                                    : (int64_t)b * c.max_pages_per_seq + pg;
  if (phys < 0 || phys >= c.num_pages) {
    set_flag(flag, KVQ_FLAG_PAGE_OOB);
    return nullptr;
  }
  const int64_t group_bytes = (int64_t)G * (9 * D / 8);
  ls = slot & (G - 1);
  const int64_t off = (((int64_t)phys * c.num_kv_heads + h) * (c.page_size >> lg_g) + (slot >> lg_g)) * group_bytes;
  if (!KVQ_IN(h >= 0 && h < c.num_kv_heads && off >= 0 &&
                  off + group_bytes <= c.num_pages * (int64_t)c.num_kv_heads * c.page_size * (9 * D / 8),
              flag))
    return nullptr;
  return static_cast<uint8_t*>(c.data) + off;
}

// K item: blocks [j0, j0 + kAppendBlocksK) of one token (src = its bf16 row of
// kv head h, at channel 16 * j0), into slot ls of group grp.
template <int D, bool NV>
__device__ __forceinline__ void append_k_item(const kvq_cache& c, uint8_t* grp, int ls, int h, int j0,
                                              const uint16_t* src, int32_t* flag) {
  constexpr int NB = D / 16;
  constexpr int BK = kAppendBlocksK;
  const int G = c.page_size < 128 ? c.page_size : 128;
  uint32_t codes[2 * BK];
  uint32_t scales = 0;
  if constexpr (NV) {
    const float S = __ldg(static_cast<const float*>(c.k_scale) + h);
    const bool fast = nv_fast_scale(S);
    const float R = __frcp_rn(S);
#pragma unroll
    for (int jb = 0; jb < BK; ++jb) {
      Raw16 kb;
      load_raw16(src + 16 * jb, kb);
      float y[16];
      uint32_t sb;
      uint2 q;
      if (fast && nv_quotients(kb, S, R, y, sb)) {
        const float s = e4m3_to_f32(sb);
        q = k_codes_f32(y, s, __frcp_rn(s));
      } else {
        const uint4 r4 = quantize_plain(src + 16 * jb, S);
        if (r4.w) set_flag(flag, KVQ_FLAG_NONFINITE);
        q = make_uint2(r4.x, r4.y);
        sb = r4.z;
      }
      codes[2 * jb] = q.x;
      codes[2 * jb + 1] = q.y;
      scales |= sb << (8 * jb);
    }
  } else {
    Raw16 kb[BK];
#pragma unroll
    for (int jb = 0; jb < BK; ++jb) load_raw16(src + 16 * jb, kb[jb]);
#pragma unroll
    for (int jb = 0; jb < BK; ++jb) {
      uint32_t sb;
      uint2 q;
      if (kb[jb].finite) {
        sb = block_scale_byte(kb[jb].amax);
        const float s = e4m3_to_f32(sb);
        q = k_codes_finite(kb[jb].w, s, scale_recip(s));
      } else {
        set_flag(flag, KVQ_FLAG_NONFINITE);
        const uint4 r4 = quantize_plain(src + 16 * jb, 1.0f);
        q = make_uint2(r4.x, r4.y);
        sb = r4.z;
      }
      codes[2 * jb] = q.x;
      codes[2 * jb + 1] = q.y;
      scales |= sb << (8 * jb);
    }
  }
  uint8_t* cdst = grp + ls * (D / 2) + 8 * j0;
  uint8_t* sdst = grp + G * (D / 2) + ls * NB + j0;
  if constexpr (BK == 1) {
    *reinterpret_cast<uint2*>(cdst) = make_uint2(codes[0], codes[1]);
    *sdst = (uint8_t)scales;
  } else {
#pragma unroll
    for (int q = 0; q < BK / 2; ++q)
      reinterpret_cast<uint4*>(cdst)[q] = make_uint4(codes[4 * q], codes[4 * q + 1], codes[4 * q + 2], codes[4 * q + 3]);
    if constexpr (BK == 2) *reinterpret_cast<uint16_t*>(sdst) = (uint16_t)scales;
    else *reinterpret_cast<uint32_t*>(sdst) = scales;
  }
}

// V item: block j0 of the token pair (pos, pos + 1) (pos even, slot ls of
// group grp even); mine0 / mine1 say which of the two tokens are new (src0 /
// src1 their bf16 rows of kv head h at channel 16 * j0).  A code byte holds
// both tokens' nibbles, so when only one token is new the other's nibbles
// and scale are kept (read-modify-write, one writer per pair).
template <int D, bool NV>
__device__ __forceinline__ void append_v_item(const kvq_cache& c, uint8_t* grp, int ls, int h, int j0, bool mine0,
                                              bool mine1, const uint16_t* src0, const uint16_t* src1,
                                              int32_t* flag) {
  constexpr int NB = D / 16;
  constexpr int BV = kAppendBlocksV;
  const int G = c.page_size < 128 ? c.page_size : 128;
  // V: token pair row ls/2 of the group
  Raw16 vb[2][BV];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const bool m = hf ? mine1 : mine0;
    const uint16_t* src = hf ? src1 : src0;
#pragma unroll
    for (int jb = 0; jb < BV; ++jb) {
      if (m) {
        load_raw16(src + 16 * jb, vb[hf][jb]);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) vb[hf][jb].w[q] = 0u;
        vb[hf][jb].amax = 0.0f;
        vb[hf][jb].finite = true;
      }
    }
  }
  const int pr = ls >> 1;
  uint8_t* vsc = grp + (int64_t)G * (D + NB) + pr * 2 * NB + 2 * j0;
  uint64_t sc = 0;  // scale bytes of the item's blocks, token 0 in the even bytes
#pragma unroll
  for (int jb = 0; jb < BV; ++jb) {
    const int j = j0 + jb;
    const int64_t vblk = (D == 64) ? (int64_t)G * (D / 2 + NB) + pr * D + 8 * ((2 * j) ^ (((pr >> 1) & 1) << 2))
                                   : (int64_t)G * (D / 2 + NB) + pr * D + 16 * (j ^ ((pr & 3) << 1));
    uint4* dst = reinterpret_cast<uint4*>(grp + vblk);
    uint4 codes;
    uint32_t sb0 = 0, sb1 = 0;
    const float S = NV ? __ldg(static_cast<const float*>(c.v_scale) + h) : 1.0f;
    float y0[16], y1[16];
    if (!NV && vb[0][jb].finite && vb[1][jb].finite) {
      sb0 = block_scale_byte(vb[0][jb].amax);
      sb1 = block_scale_byte(vb[1][jb].amax);
      const float s0 = e4m3_to_f32(sb0), s1 = e4m3_to_f32(sb1);
      codes = v_pair_codes_finite(vb[0][jb].w, s0, scale_recip(s0), vb[1][jb].w, s1, scale_recip(s1));
    } else if (NV && nv_fast_scale(S) && nv_quotients(vb[0][jb], S, __frcp_rn(S), y0, sb0) &&
               nv_quotients(vb[1][jb], S, __frcp_rn(S), y1, sb1)) {
      const float s0 = e4m3_to_f32(sb0), s1 = e4m3_to_f32(sb1);
      codes = v_pair_codes_f32(y0, s0, __frcp_rn(s0), y1, s1, __frcp_rn(s1));
    } else {
      uint64_t lo = 0, hi = 0;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        if (!(hf ? mine1 : mine0)) continue;
        const uint16_t* vsrc = (hf ? src1 : src0) + 16 * jb;
        const uint4 q = quantize_plain(vsrc, S);
        if (q.w) set_flag(flag, KVQ_FLAG_NONFINITE);
        lo |= spread_nibbles(q.x) << (4 * hf);
        hi |= spread_nibbles(q.y) << (4 * hf);
        (hf ? sb1 : sb0) = q.z;
      }
      codes = make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
    }
    sc |= (uint64_t)(sb0 | (sb1 << 8)) << (16 * jb);
    if (!(mine0 && mine1)) {
      // keep the nibbles of the token that is not new
      const uint32_t keep = mine0 ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
      const uint4 old = *dst;
      codes.x |= old.x & keep;
      codes.y |= old.y & keep;
      codes.z |= old.z & keep;
      codes.w |= old.w & keep;
    }
    *dst = codes;
  }
  if (mine0 && mine1) {
    if constexpr (BV == 4) *reinterpret_cast<uint2*>(vsc) = make_uint2((uint32_t)sc, (uint32_t)(sc >> 32));
    else if constexpr (BV == 2) *reinterpret_cast<uint32_t*>(vsc) = (uint32_t)sc;
    else *reinterpret_cast<uint16_t*>(vsc) = (uint16_t)sc;
  } else {
    // keep the scales of the token that is not new
    const int hf = mine0 ? 0 : 1;
#pragma unroll
    for (int jb = 0; jb < BV; ++jb) vsc[2 * jb + hf] = (uint8_t)(sc >> (16 * jb + 8 * hf));
  }
}

}  // namespace
}  // namespace kvq
