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

__global__ void __launch_bounds__(256) append_fp4_kernel(const kvq_cache c, int32_t batch, int32_t n_new,
                                                         const int32_t* __restrict__ start_pos,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, int32_t* flag) {
  const int nblk = c.head_dim >> 4;
  const int Hkv = c.num_kv_heads;
  const int P = c.page_size;
  const int64_t total = (int64_t)batch * n_new * Hkv * nblk;
  uint8_t* kc = static_cast<uint8_t*>(c.k_codes);
  uint8_t* vc = static_cast<uint8_t*>(c.v_codes);
  uint8_t* ks = static_cast<uint8_t*>(c.k_scales);
  uint8_t* vs = static_cast<uint8_t*>(c.v_scales);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % nblk);
    int64_t r = i / nblk;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int t = (int)(r % n_new);
    const int b = (int)(r / n_new);
    const int32_t sp = __ldg(start_pos + b);
    if (sp < 0) {
      set_flag(flag, KVQ_FLAG_BAD_LENGTH);
      continue;
    }
    const int64_t pos = (int64_t)sp + t;
    const int64_t pg = pos / P;
    const int slot = (int)(pos % P);
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
    const int64_t row = (phys * Hkv + h) * P + slot;
    const Block16 kb = load_bf16x16(k + i * 16);
    const Block16 vb = load_bf16x16(v + i * 16);
    if (!kb.finite || !vb.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
    uint32_t ksb, vsb;
    const uint2 kq = quantize_block(kb, ksb);
    const uint2 vq = quantize_block(vb, vsb);
    *reinterpret_cast<uint2*>(kc + row * (c.head_dim >> 1) + 8 * j) = kq;
    *reinterpret_cast<uint2*>(vc + row * (c.head_dim >> 1) + 8 * j) = vq;
    ks[row * nblk + j] = (uint8_t)ksb;
    vs[row * nblk + j] = (uint8_t)vsb;
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
  const float* ksc = static_cast<const float*>(c.k_scales);
  const float* vsc = static_cast<const float*>(c.v_scales);
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
      uint8_t* base = static_cast<uint8_t*>(side ? c.v_codes : c.k_codes);
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
    static_cast<float*>(side ? c.v_scales : c.k_scales)[h] = s;
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
  const int64_t work = (int64_t)batch * n_new * cache->num_kv_heads * (cache->head_dim / 16);
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
