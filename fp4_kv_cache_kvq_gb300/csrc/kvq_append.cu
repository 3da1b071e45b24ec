// kvq_append.cu -- quantise-on-append into the FP4 paged cache and the FP8
// window cache, and the FP8 per-head scale calibration.
//
// FP4 block quantiser ("Quantising the KV cache", section "Code"): for each
// 16-channel block of one token and one kv head, s = RNE_e4m3(amax / 6)
// saturating (a zero scale becomes the E4M3 min subnormal 2^-9), then each
// value becomes RNE_e2m1(v / s) saturating, with both divisions IEEE fp32 and
// the sign of every value kept in its nibble.  Two codes per byte, even
// channel in the low nibble; one E4M3 scale byte per block.
//
// FP8 window ("Week 6 -- FP4 KV Caches and Bounded Replay", "Overview": the
// SWA KV stays FP8): code = RNE_e4m3(x / s_h) saturating with one fp32 scale
// per kv head, s_h = amax / 448 over a calibration window (1 if amax == 0).
//
// Work decomposition: one thread per 16-value block (32 B of bf16 read with two
// 16-byte loads, 8 code bytes + 1 scale byte written); consecutive threads take
// consecutive blocks of the input, so loads and stores are coalesced.
#include "kvq_common.cuh"
#include "kvq_host.cuh"

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

// Spread 8 nibbles (nibble c at bits 4c) to 8 bytes (nibble c in the low half
// of byte c).
__device__ __forceinline__ uint64_t spread_nibbles(uint32_t w) {
  uint64_t x = w;
  x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
  x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
  x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
  return x;
}

// Work items: first one per (sequence, new token, kv head, 16-channel block)
// for K, then one per (sequence, token pair, kv head, block) for V.  A V item
// owns the 16 interleaved bytes of its pair, so when only one token of the pair
// is new it keeps the other token's nibbles (read-modify-write, one writer).
__global__ void __launch_bounds__(256) append_fp4_kernel(const kvq_cache c, int32_t batch, int32_t n_new,
                                                         const int32_t* __restrict__ start_pos,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, int32_t* flag) {
  const Fp4Layout L(c.head_dim, c.page_size);
  const int nb = L.nb;
  const int Hkv = c.num_kv_heads;
  const int D = c.head_dim;
  const int npair = n_new / 2 + 1;  // token pairs a call of n_new tokens can touch
  const int64_t nk = (int64_t)batch * n_new * Hkv * nb;
  const int64_t total = nk + (int64_t)batch * npair * Hkv * nb;
  uint8_t* pool = static_cast<uint8_t*>(c.data);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_k = i < nk;
    const int64_t e = is_k ? i : i - nk;
    const int j = (int)(e % nb);
    int64_t r = e / nb;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int per = is_k ? n_new : npair;
    const int t = (int)(r % per);
    const int b = (int)(r / per);
    const int32_t sp = __ldg(start_pos + b);
    if (sp < 0) {
      if (is_k) set_flag(flag, KVQ_FLAG_BAD_LENGTH);
      continue;
    }
    // first position handled by this item (K: the token, V: the pair's even token)
    const int64_t pos = is_k ? (int64_t)sp + t : 2 * (((int64_t)sp >> 1) + t);
    if (!is_k && pos >= (int64_t)sp + n_new) continue;
    const int64_t pg = pos / L.P;
    const int slot = (int)(pos % L.P);
    if (pg >= c.max_pages_per_seq) {
      set_flag(flag, KVQ_FLAG_PAGE_OOB);
      continue;
    }
    const int64_t phys = c.page_table ? (int64_t)__ldg(c.page_table + (int64_t)b * c.max_pages_per_seq + pg)
                                      : (int64_t)b * c.max_pages_per_seq + pg;
    if (phys < 0 || phys >= c.num_pages) {
      set_flag(flag, KVQ_FLAG_PAGE_OOB);
      continue;
    }
    uint8_t* grp = pool + L.group(phys, Hkv, h, slot);
    const int ls = slot % L.G;
    if (is_k) {
      const Block16 kb = load_bf16x16(k + (((int64_t)b * n_new + t) * Hkv + h) * D + 16 * j);
      if (!kb.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
      uint32_t sb;
      const uint2 q = quantize_block(kb, sb);
      *reinterpret_cast<uint2*>(grp + (int64_t)ls * (D / 2) + 8 * j) = q;
      grp[L.k_scales() + (int64_t)ls * nb + j] = (uint8_t)sb;
    } else {
      uint4* dst = reinterpret_cast<uint4*>(grp + L.v_block(ls >> 1, j));
      uint4 old = make_uint4(0u, 0u, 0u, 0u);
      uint64_t lo = 0, hi = 0;  // interleaved bytes of channels 0-7 and 8-15
      uint64_t keep_lo = 0, keep_hi = 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int64_t p = pos + half;
        const bool mine = p >= sp && p < (int64_t)sp + n_new;
        if (mine) {
          const int tt = (int)(p - sp);
          const Block16 vb = load_bf16x16(v + (((int64_t)b * n_new + tt) * Hkv + h) * D + 16 * j);
          if (!vb.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
          uint32_t sb;
          const uint2 q = quantize_block(vb, sb);
          lo |= spread_nibbles(q.x) << (4 * half);
          hi |= spread_nibbles(q.y) << (4 * half);
          grp[L.v_scale(ls + half, j)] = (uint8_t)sb;
        } else {
          const uint64_t m = half ? 0xF0F0F0F0F0F0F0F0ull : 0x0F0F0F0F0F0F0F0Full;
          keep_lo |= m;
          keep_hi |= m;
        }
      }
      if (keep_lo) old = *dst;
      lo |= (((uint64_t)old.y << 32) | old.x) & keep_lo;
      hi |= (((uint64_t)old.w << 32) | old.z) & keep_hi;
      *dst = make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
    }
  }
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

__global__ void __launch_bounds__(256) append_fp8_kernel(const kvq_cache c, int32_t batch, int32_t n_new,
                                                         const int32_t* __restrict__ start_pos,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, int32_t* flag) {
  const int nblk = c.head_dim >> 4;
  const int Hkv = c.num_kv_heads;
  const int W = c.page_size;
  const int64_t total = (int64_t)batch * n_new * Hkv * nblk;
  const float* ksc = static_cast<const float*>(c.k_scale);
  const float* vsc = static_cast<const float*>(c.v_scale);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % nblk);
    int64_t r = i / nblk;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int t = (int)(r % n_new);
    const int b = (int)(r / n_new);
    if (t < n_new - W) continue;  // a later token of this call takes the same slot
    const int32_t sp = __ldg(start_pos + b);
    if (sp < 0) {
      set_flag(flag, KVQ_FLAG_BAD_LENGTH);
      continue;
    }
    const int slot = (int)(((int64_t)sp + t) % W);
    const int64_t dst = (((int64_t)b * Hkv + h) * W + slot) * c.head_dim + 16 * j;
    const float sk = __ldg(ksc + h), sv = __ldg(vsc + h);
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const Block16 blk = load_bf16x16((side ? v : k) + i * 16);
      if (!blk.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
      const float s = side ? sv : sk;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = e4m3_pair(blk.x[4 * q], blk.x[4 * q + 1], s) | (e4m3_pair(blk.x[4 * q + 2], blk.x[4 * q + 3], s) << 16);
      uint8_t* base = static_cast<uint8_t*>(side ? c.v_data : c.data);
      *reinterpret_cast<uint4*>(base + dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// One CTA per (kv head, K/V): amax over every value of that head, then
// s_h = amax / 448 (IEEE fp32), 1 if amax == 0.
__global__ void __launch_bounds__(256) fp8_scales_kernel(const kvq_cache c, int64_t rows,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, int32_t* flag) {
  const int h = blockIdx.x;
  const int side = blockIdx.y;
  const uint16_t* src = side ? v : k;
  const int D = c.head_dim;
  const int Hkv = c.num_kv_heads;
  const int per_row = D >> 4;
  float amax = 0.0f;
  bool finite = true;
  for (int64_t i = threadIdx.x; i < rows * per_row; i += blockDim.x) {
    const int64_t r = i / per_row;
    const int j = (int)(i % per_row);
    const Block16 b = load_bf16x16(src + (r * Hkv + h) * D + 16 * j);
    finite &= b.finite;
#pragma unroll
    for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(b.x[q]));
  }
  __shared__ float red[32];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  if (!finite) atomicOr(&bad, 1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
    if (bad) set_flag(flag, KVQ_FLAG_NONFINITE);
    const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
    static_cast<float*>(side ? c.v_scale : c.k_scale)[h] = s;
  }
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_append(const kvq_cache* cache, int32_t batch, int32_t n_new, const int32_t* d_start_pos,
                                 const void* k, const void* v, int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 0 || n_new < 0) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (batch == 0 || n_new == 0) return KVQ_OK;
  if (d_start_pos == nullptr || k == nullptr || v == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(k, 16) || !aligned_to(v, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  const int64_t work = (int64_t)batch * (n_new + n_new / 2 + 1) * cache->num_kv_heads * (cache->head_dim / 16);
  const unsigned grid = grid_for(work, 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cache->format == KVQ_FORMAT_FP4_E2M1_E4M3_G16) {
    append_fp4_kernel<<<grid, 256, 0, s>>>(*cache, batch, n_new, d_start_pos, static_cast<const uint16_t*>(k),
                                           static_cast<const uint16_t*>(v), d_err_flag);
  } else {
    append_fp8_kernel<<<grid, 256, 0, s>>>(*cache, batch, n_new, d_start_pos, static_cast<const uint16_t*>(k),
                                           static_cast<const uint16_t*>(v), d_err_flag);
  }
  return launch_status();
}

extern "C" kvq_status kvq_fp8_set_scales(const kvq_cache* cache, int32_t batch, int32_t n, const void* k,
                                         const void* v, int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 0 || n < 0) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (cache->format != KVQ_FORMAT_FP8_E4M3_HEAD) return KVQ_ERR_INVALID_ARGUMENT;
  if ((int64_t)batch * n > 0 && (k == nullptr || v == nullptr)) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(k, 16) || !aligned_to(v, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  dim3 grid(cache->num_kv_heads, 2);
  fp8_scales_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      *cache, (int64_t)batch * n, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), d_err_flag);
  return launch_status();
}

extern "C" const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

extern "C" int32_t kvq_version(void) { return KVQ_VERSION; }

extern "C" size_t kvq_fp4_pool_bytes(int64_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim) {
  if (num_pages < 0 || num_kv_heads < 1 || !is_pow2_page(page_size) ||
      (head_dim != 64 && head_dim != 128 && head_dim != 256))
    return 0;
  return (size_t)num_pages * (size_t)num_kv_heads * (size_t)page_size * 9u * (size_t)head_dim / 8u;
}
