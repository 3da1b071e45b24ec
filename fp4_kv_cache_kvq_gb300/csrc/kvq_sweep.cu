// kvq_sweep.cu -- the bit-width / layout sweep: fake quantisation (quantise,
// then dequantise) of a K or V tensor in the formats that the results table
// of "Quantising the KV cache" compares, and a dense decode attention with
// fp64 accumulation that measures what each format does to the output.
//
// Formats (the pages give their storage cost -- section "Maths", b + s/g bits
// -- and the FP4 rounding -- section "Code" -- but not the INT rounding; the
// readings below are the plainest ones the rest supports):
//   FP8 E4M3, one scale per tensor: s = amax / 448 over the whole tensor in
//     fp32 (1 when amax == 0), code RNE_e4m3(x / s) saturating, x^ = e4m3(c)*s.
//   INT-b, symmetric, one FP16 scale per group: s = FP16_RNE(amax / qmax) with
//     qmax = 2^(b-1) - 1 and an fp32 division, saturating at 65504, a zero
//     scale replaced by the smallest FP16 subnormal 2^-24; code
//     clamp(RNE(x / s), -qmax, qmax) with an fp32 division (NaN -> 0);
//     x^ = code * s.  A per-token group is one token's head_dim channels of
//     one head, a per-channel group one channel of one head over the tensor's
//     tokens (section "Per token or per channel?").
//   FP4 E2M1 with an E4M3 scale per 16 channels: the cache's block quantiser.
#include <cuda_fp16.h>

#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_host.cuh"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

// FP16 group scale of an INT-b group (see the file comment); returns it and
// its bit pattern.
__device__ __forceinline__ float int_group_scale(float amax, int qmax, uint16_t& bits) {
  const float t = fminf(__fdiv_rn(amax, (float)qmax), 65504.0f);
  uint16_t b = __half_as_ushort(__float2half_rn(t));
  if ((b & 0x7FFFu) == 0) b = 0x0001u;
  bits = b;
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ int int_code(float x, float s, int qmax) {
  const float y = __fdiv_rn(x, s);
  if (isnan(y)) return 0;
  if (y >= (float)qmax) return qmax;
  if (y <= -(float)qmax) return -qmax;
  return __float2int_rn(y);
}

__device__ __forceinline__ float bf16_at(const uint16_t* p) { return __uint_as_float((uint32_t)*p << 16); }

// INT-b per token: one warp per group of d channels.
__global__ void __launch_bounds__(256) int_per_token_kernel(const uint16_t* __restrict__ x, int64_t groups, int d,
                                                            int qmax, float* __restrict__ xh, int8_t* codes,
                                                            uint16_t* scales, int32_t* flag) {
  const int64_t gidx = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gidx >= groups) return;
  const uint16_t* row = x + gidx * d;
  float amax = 0.0f;
  bool bad = false;
  for (int c = lane; c < d; c += 32) {
    const float v = bf16_at(row + c);
    bad |= !isfinite(v);
    amax = fmaxf(amax, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  bad = __any_sync(0xFFFFFFFFu, bad);
  uint16_t sb;
  const float s = int_group_scale(amax, qmax, sb);
  for (int c = lane; c < d; c += 32) {
    const int q = int_code(bf16_at(row + c), s, qmax);
    xh[gidx * d + c] = (float)q * s;
    if (codes) codes[gidx * d + c] = (int8_t)q;
  }
  if (lane == 0) {
    if (scales) scales[gidx] = sb;
    if (bad) set_flag(flag, KVQ_FLAG_NONFINITE);
  }
}

// INT-b per channel: one thread per (sequence, head, channel), over the tokens.
__global__ void __launch_bounds__(256) int_per_channel_kernel(const uint16_t* __restrict__ x, int batch, int tokens,
                                                              int heads, int d, int qmax, float* __restrict__ xh,
                                                              int8_t* codes, uint16_t* scales, int32_t* flag) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)batch * heads * d) return;
  const int c = (int)(i % d);
  const int h = (int)((i / d) % heads);
  const int64_t b = i / ((int64_t)d * heads);
  const int64_t base = (b * tokens * heads + h) * d + c, stride = (int64_t)heads * d;
  float amax = 0.0f;
  bool bad = false;
  for (int t = 0; t < tokens; ++t) {
    const float v = bf16_at(x + base + t * stride);
    bad |= !isfinite(v);
    amax = fmaxf(amax, fabsf(v));
  }
  uint16_t sb;
  const float s = int_group_scale(amax, qmax, sb);
  for (int t = 0; t < tokens; ++t) {
    const int q = int_code(bf16_at(x + base + t * stride), s, qmax);
    xh[base + t * stride] = (float)q * s;
    if (codes) codes[base + t * stride] = (int8_t)q;
  }
  if (scales) scales[(b * heads + h) * d + c] = sb;
  if (bad) set_flag(flag, KVQ_FLAG_NONFINITE);
}

// FP8 per tensor, pass 1: amax over every value, as the bit pattern of |x|
// (for non-negative floats the unsigned order is the numeric order; a NaN
// sorts above every number and propagates).
__global__ void __launch_bounds__(256) amax_bits_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                        unsigned int* amax_bits) {
  unsigned int m = 0u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    m = max(m, ((uint32_t)x[i] << 16) & 0x7FFFFFFFu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, m);
}

// FP8 per tensor, pass 2: one thread per 16 values.
__global__ void __launch_bounds__(256) fp8_tensor_kernel(const uint16_t* __restrict__ x, int64_t blocks,
                                                         float* scale_pair, float* __restrict__ xh, int8_t* codes,
                                                         int32_t* flag) {
  const float amax = __uint_as_float(*reinterpret_cast<const volatile unsigned int*>(scale_pair));
  const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) scale_pair[1] = s;
  if (i >= blocks) return;
  const Block16 blk = load_bf16x16(x + i * 16);
  if (!blk.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t pr = e4m3_pair(blk.x[2 * j], blk.x[2 * j + 1], s);
    const float2 f = f16x2_to_float2(f16x2_from_e4m3x2(pr));
    xh[i * 16 + 2 * j] = f.x * s;
    xh[i * 16 + 2 * j + 1] = f.y * s;
    if (codes) {
      codes[i * 16 + 2 * j] = (int8_t)(pr & 0xFFu);
      codes[i * 16 + 2 * j + 1] = (int8_t)(pr >> 8);
    }
  }
}

// FP4 E2M1 + E4M3 per 16: one thread per block.
__global__ void __launch_bounds__(256) fp4_block_kernel(const uint16_t* __restrict__ x, int64_t blocks,
                                                        float* __restrict__ xh, int8_t* codes, uint8_t* scales,
                                                        int32_t* flag) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= blocks) return;
  const Block16 blk = load_bf16x16(x + i * 16);
  if (!blk.finite) set_flag(flag, KVQ_FLAG_NONFINITE);
  uint32_t sb;
  const uint2 q = quantize_block(blk, sb);
  const float s = e4m3_to_f32(sb);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t byte = ((j < 4 ? q.x : q.y) >> (8 * (j & 3))) & 0xFFu;
    const float2 f = f16x2_to_float2(f16x2_from_e2m1x2(byte));
    xh[i * 16 + 2 * j] = f.x * s;
    xh[i * 16 + 2 * j + 1] = f.y * s;
    if (codes) {
      codes[i * 16 + 2 * j] = (int8_t)(byte & 0xFu);
      codes[i * 16 + 2 * j + 1] = (int8_t)(byte >> 4);
    }
  }
  if (scales) scales[i] = (uint8_t)sb;
}

// ------------------------------------------------------------------ dense attention
constexpr int kDenseThreads = 256;
constexpr int kDenseMaxTokens = 16384;

__device__ __forceinline__ void block_argmax(double& v, int& idx, double* rv, int* ri) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
    if (v2 > v || (v2 == v && i2 < idx)) {
      v = v2;
      idx = i2;
    }
  }
  __syncthreads();
  if (lane == 0) {
    rv[warp] = v;
    ri[warp] = idx;
  }
  __syncthreads();
  v = rv[0];
  idx = ri[0];
  for (int w = 1; w < kDenseThreads / 32; ++w)
    if (rv[w] > v || (rv[w] == v && ri[w] < idx)) {
      v = rv[w];
      idx = ri[w];
    }
}

__device__ __forceinline__ double block_sum(double v, double* rv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if (lane == 0) rv[warp] = v;
  __syncthreads();
  double s = 0.0;
  for (int w = 0; w < kDenseThreads / 32; ++w) s += rv[w];
  return s;
}

// One CTA per (sequence, query head): out = softmax(scale * q.K^T) V with
// every product, the softmax and the sums in fp64; top = the position with
// the largest score (the lowest one on a tie).
__global__ void __launch_bounds__(kDenseThreads) attn_dense_kernel(int tokens, int hq, int hkv, int d,
                                                                   const uint16_t* __restrict__ q,
                                                                   const float* __restrict__ k,
                                                                   const float* __restrict__ v, double scale,
                                                                   float* __restrict__ out, int32_t* top) {
  extern __shared__ double dsm[];
  double* qs = dsm;             // [d]
  double* sc = qs + d;          // [tokens]
  double* rv = sc + tokens;     // [warps]
  int* ri = reinterpret_cast<int*>(rv + kDenseThreads / 32);
  const int b = blockIdx.x / hq, hh = blockIdx.x % hq;
  const int kh = hh / (hq / hkv);
  const int tid = threadIdx.x;
  for (int c = tid; c < d; c += kDenseThreads) qs[c] = (double)bf16_at(q + ((int64_t)b * hq + hh) * d + c);
  __syncthreads();
  double mx = -INFINITY;
  int arg = 0x7FFFFFFF;
  for (int t = tid; t < tokens; t += kDenseThreads) {
    const float* kr = k + (((int64_t)b * tokens + t) * hkv + kh) * d;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc = fma(qs[c], (double)kr[c], acc);
    acc *= scale;
    sc[t] = acc;
    if (acc > mx) {
      mx = acc;
      arg = t;
    }
  }
  block_argmax(mx, arg, rv, ri);
  double l = 0.0;
  for (int t = tid; t < tokens; t += kDenseThreads) {
    const double e = exp(sc[t] - mx);
    sc[t] = e;
    l += e;
  }
  l = block_sum(l, rv);  // its barriers also publish sc[]
  for (int c = tid; c < d; c += kDenseThreads) {
    double o = 0.0;
    for (int t = 0; t < tokens; ++t) o = fma(sc[t], (double)v[(((int64_t)b * tokens + t) * hkv + kh) * d + c], o);
    out[((int64_t)b * hq + hh) * d + c] = tokens > 0 ? (float)(o / l) : 0.0f;
  }
  if (tid == 0 && top) top[(int64_t)b * hq + hh] = tokens > 0 ? arg : -1;
}

int dense_smem_bytes(int d, int tokens) {
  return (d + tokens + kDenseThreads / 32) * (int)sizeof(double) + kDenseThreads / 32 * (int)sizeof(int);
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_fake_quant(int32_t layout, int32_t bits, int32_t batch, int32_t tokens, int32_t heads,
                                     int32_t head_dim, const void* x, float* x_hat, int8_t* codes, void* scales,
                                     int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 0 || tokens < 0 || heads < 1 || head_dim < 16 || head_dim % 16 != 0) return KVQ_ERR_INVALID_ARGUMENT;
  const int64_t n = (int64_t)batch * tokens * heads * head_dim;
  if (n == 0) return KVQ_OK;
  if (x == nullptr || x_hat == nullptr || !aligned_to(x, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  switch (layout) {
    case KVQ_LAYOUT_FP8_TENSOR: {
      if (bits != 8 || scales == nullptr || !aligned_to(scales, 8)) return KVQ_ERR_INVALID_ARGUMENT;
      float* sp = static_cast<float*>(scales);
      if (cudaMemsetAsync(sp, 0, sizeof(float), s) != cudaSuccess) return KVQ_ERR_CUDA;
      const unsigned g1 = (unsigned)std::min<int64_t>(grid_for(n, 256), 8 * (int64_t)std::max(1, device_sm_count()));
      amax_bits_kernel<<<g1, 256, 0, s>>>(xs, n, reinterpret_cast<unsigned int*>(sp));
      fp8_tensor_kernel<<<grid_for(n / 16, 256), 256, 0, s>>>(xs, n / 16, sp, x_hat, codes, d_err_flag);
      return launch_status();
    }
    case KVQ_LAYOUT_INT_PER_TOKEN:
    case KVQ_LAYOUT_INT_PER_CHANNEL: {
      if (bits < 2 || bits > 8) return KVQ_ERR_INVALID_ARGUMENT;
      const int qmax = (1 << (bits - 1)) - 1;
      uint16_t* sc = static_cast<uint16_t*>(scales);
      if (layout == KVQ_LAYOUT_INT_PER_TOKEN) {
        const int64_t groups = (int64_t)batch * tokens * heads;
        int_per_token_kernel<<<grid_for(groups * 32, 256), 256, 0, s>>>(xs, groups, head_dim, qmax, x_hat, codes,
                                                                          sc, d_err_flag);
      } else {
        const int64_t threads = (int64_t)batch * heads * head_dim;
        int_per_channel_kernel<<<grid_for(threads, 256), 256, 0, s>>>(xs, batch, tokens, heads, head_dim, qmax,
                                                                        x_hat, codes, sc, d_err_flag);
      }
      return launch_status();
    }
    case KVQ_LAYOUT_FP4_G16:
      if (bits != 4) return KVQ_ERR_INVALID_ARGUMENT;
      fp4_block_kernel<<<grid_for(n / 16, 256), 256, 0, s>>>(xs, n / 16, x_hat, codes, static_cast<uint8_t*>(scales),
                                                              d_err_flag);
      return launch_status();
    default:
      return KVQ_ERR_INVALID_ARGUMENT;
  }
}

extern "C" kvq_status kvq_attn_dense(int32_t batch, int32_t tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, const void* q, const float* k, const float* v,
                                     float softmax_scale, float* out, int32_t* top, kvq_stream stream) {
  if (batch < 0 || tokens < 0 || num_kv_heads < 1 || num_q_heads < num_kv_heads ||
      num_q_heads % num_kv_heads != 0 || head_dim < 1 || !(softmax_scale > 0.0f))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (tokens > kDenseMaxTokens || head_dim > 512) return KVQ_ERR_UNSUPPORTED;
  if (batch == 0) return KVQ_OK;
  if (q == nullptr || out == nullptr || (tokens > 0 && (k == nullptr || v == nullptr))) return KVQ_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  static DeviceOnce attr_set;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(attn_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dense_smem_bytes(512, kDenseMaxTokens)) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  attn_dense_kernel<<<(unsigned)(batch * num_q_heads), kDenseThreads, dense_smem_bytes(head_dim, tokens), s>>>(
      tokens, num_q_heads, num_kv_heads, head_dim, static_cast<const uint16_t*>(q), k, v, (double)softmax_scale,
      out, top);
  return launch_status();
}
