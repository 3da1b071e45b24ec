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
// FP4 work decomposition: one thread per 2 blocks of one token (K) or per
// block of one token pair (V, whose code bytes interleave the two tokens);
// consecutive threads take consecutive spans of the input, so loads and
// stores coalesce.  Finite blocks take a division-free path whose codes equal
// those of the IEEE divisions (reciprocal quotient plus one exact residual
// correction, argued at block_quotient); blocks holding Inf or NaN take the
// plain IEEE-division quantiser.
#include "kvq_append.cuh"
#include "kvq_common.cuh"
#include "kvq_host.cuh"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

// n / d for n < 2^31 without a hardware divide: (umulhi(n, mul) + n) >> shift
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up variant with a 33-bit multiplier).
struct DivU32 {
  uint32_t mul, shift;
  static DivU32 make(uint32_t d) {
    if (d <= 1u) return DivU32{0u, 0u};
    uint32_t sh = 0;
    while ((1ull << sh) < d) ++sh;
    return DivU32{(uint32_t)((((1ull << 32) * ((1ull << sh) - d)) / d) + 1u), sh};
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, mul) + n) >> shift; }
};

// CTAs per SM the register budget is set for (blocks per item:
// kvq_append.cuh).  Six CTAs of 256 threads cap the kernel at 40 registers,
// with a few spilled bytes, but keep 50% more loads in flight than four
// (63 registers, no spills): measured on the 16 x 16384-token prefill,
// 258 -> 240 us (FP4) and 312 -> 291 us (NVFP4); eight CTAs (32 registers,
// 150-250 spilled bytes) ran at 266 us.
constexpr int kAppendMinCtas = 6;

// Work items, one thread each: one per (sequence, new token, kv head, group
// of kAppendBlocksK blocks) for K, in the first k_ctas CTAs; then one per
// (sequence, token pair, kv head, group of kAppendBlocksV blocks) for V.  A V item owns the interleaved
// bytes of its pair, so when only one token of the pair is new it keeps the
// other token's nibbles (read-modify-write, one writer).  Consecutive threads
// take consecutive spans of the input; the row, page and address arithmetic
// is done once per item, not once per block.  Indices are 32-bit;
// the host splits the batch so that every launch's item count fits.
// NV: an NVFP4 cache (codes of x / S_h from nv_quotients; blocks it refuses
// take the IEEE-division quantiser).
template <int D, bool NV>
__global__ void __launch_bounds__(256, kAppendMinCtas) append_fp4_kernel(const kvq_cache c, int32_t b_begin, uint32_t k_items,
                                                         uint32_t v_items, uint32_t k_ctas, DivU32 div_hkv,
                                                         DivU32 div_k_per, DivU32 div_v_per, int32_t n_new,
                                                         const int32_t* __restrict__ start_pos, int32_t sp_offset,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, int32_t* flag) {
  constexpr int NB = D / 16;
  constexpr int BK = kAppendBlocksK, BV = kAppendBlocksV;
  constexpr int NQK = NB / BK, NQV = NB / BV;  // items per (token, head) row
  // a decode launched as a programmatic dependent of this append may be
  // scheduled now; it waits for this grid before copying any pool bytes
  grid_launch_dependents();
  const bool is_k = blockIdx.x < k_ctas;
  const uint32_t i = (is_k ? blockIdx.x : blockIdx.x - k_ctas) * 256u + threadIdx.x;
  if (i >= (is_k ? k_items : v_items)) return;
  const uint32_t hkv = (uint32_t)c.num_kv_heads;
  const int j0 = is_k ? (int)(i % NQK) * BK : (int)(i % NQV) * BV;
  const uint32_t r = is_k ? i / NQK : i / NQV;
  const uint32_t r2 = div_hkv.div(r);
  const int h = (int)(r - r2 * hkv);
  const uint32_t per = is_k ? (uint32_t)n_new : (uint32_t)(n_new / 2 + 1);
  const uint32_t bq = (is_k ? div_k_per : div_v_per).div(r2);
  const uint32_t t = r2 - bq * per;
  const int b = b_begin + (int)bq;
  // sp_offset -1: start_pos holds lengths that include the one new token
  // (the decode step's append); a zero length appends nothing
  const int32_t sp = __ldg(start_pos + b) + sp_offset;
  if (sp < 0) {
    if (is_k && sp < sp_offset) set_flag(flag, KVQ_FLAG_BAD_LENGTH);
    return;
  }
  // first position handled by this item (K: the token, V: the pair's even token)
  const int64_t pos = is_k ? (int64_t)sp + t : 2 * (((int64_t)sp >> 1) + t);
  const int64_t end = (int64_t)sp + n_new;
  if (!is_k && pos >= end) return;
  int ls = 0;
  uint8_t* grp = fp4_group<D>(c, b, pos, h, ls, flag);
  if (grp == nullptr) return;
  const int64_t row = (int64_t)b * n_new;  // first input row of sequence b
  // (bounds-checked build: the item's input rows lie inside this launch's
  // batch x n_new rows)
  if (!KVQ_IN(t < (uint32_t)n_new && (is_k || (pos - sp >= -1 && pos + 1 - sp <= n_new)), flag)) return;
  if (is_k) {
    append_k_item<D, NV>(c, grp, ls, h, j0, k + ((row + t) * hkv + h) * D + 16 * j0, flag);
    return;
  }
  // V: the pair (pos, pos + 1); a token outside this call's range keeps its bytes
  const bool mine0 = pos >= sp;
  const bool mine1 = pos + 1 < end;
  const uint16_t* src0 = v + ((row + (pos - sp)) * hkv + h) * D + 16 * j0;
  const uint16_t* src1 = v + ((row + (pos + 1 - sp)) * hkv + h) * D + 16 * j0;
  append_v_item<D, NV>(c, grp, ls, h, j0, mine0, mine1, src0, src1, flag);
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
// s_h = amax / divisor (IEEE fp32; 448 for an FP8 cache, 6 * 448 for the
// NVFP4 second level), 1 if amax == 0.
__global__ void __launch_bounds__(256) fp8_scales_kernel(const kvq_cache c, int64_t rows,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, float divisor,
                                                         int32_t* flag) {
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
    const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, divisor);
    static_cast<float*>(side ? c.v_scale : c.k_scale)[h] = s;
  }
}

}  // namespace
}  // namespace kvq

using namespace kvq;

namespace kvq {

// The FP4 / NVFP4 append launches of kvq_append (n_new tokens per sequence
// from start_pos[b] + sp_offset), shared with kvq_append_decode_attn's
// separate-append path (n_new 1, start_pos the lengths, sp_offset -1).
kvq_status launch_fp4_append(const kvq_cache* cache, int32_t batch, int32_t n_new, const int32_t* d_start_pos,
                             int32_t sp_offset, const uint16_t* k16, const uint16_t* v16, int32_t* d_err_flag,
                             cudaStream_t s) {
  const bool nv = cache->format == KVQ_FORMAT_NVFP4;
  // 32-bit item indices: one sequence's items must fit, the batch is split.
  const int64_t nqk = cache->head_dim / 16 / kAppendBlocksK;  // items per (token, head)
  const int64_t nqv = cache->head_dim / 16 / kAppendBlocksV;
  const int64_t per_seq = (int64_t)n_new * cache->num_kv_heads * nqk;
  const int64_t limit = (int64_t)1 << 30;
  if ((int64_t)n_new * cache->num_kv_heads * (cache->head_dim / 16) > limit) return KVQ_ERR_UNSUPPORTED;
  const int64_t chunk = limit / per_seq;
  for (int64_t b0 = 0; b0 < batch; b0 += chunk) {
    const int64_t bc = (batch - b0 < chunk) ? batch - b0 : chunk;
    const uint32_t k_items = (uint32_t)(bc * per_seq);
    const uint32_t v_items = (uint32_t)(bc * (n_new / 2 + 1) * cache->num_kv_heads * nqv);
    const uint32_t k_ctas = (k_items + 255u) / 256u;
    const uint32_t grid = k_ctas + (v_items + 255u) / 256u;
    const DivU32 dh = DivU32::make((uint32_t)cache->num_kv_heads);
    const DivU32 dk = DivU32::make((uint32_t)n_new);
    const DivU32 dv = DivU32::make((uint32_t)(n_new / 2 + 1));
    switch (cache->head_dim) {
      case 64:
        (nv ? append_fp4_kernel<64, true> : append_fp4_kernel<64, false>)<<<grid, 256, 0, s>>>(
            *cache, (int32_t)b0, k_items, v_items, k_ctas, dh, dk, dv, n_new, d_start_pos, sp_offset, k16, v16,
            d_err_flag);
        break;
      case 128:
        (nv ? append_fp4_kernel<128, true> : append_fp4_kernel<128, false>)<<<grid, 256, 0, s>>>(
            *cache, (int32_t)b0, k_items, v_items, k_ctas, dh, dk, dv, n_new, d_start_pos, sp_offset, k16, v16,
            d_err_flag);
        break;
      default:
        (nv ? append_fp4_kernel<256, true> : append_fp4_kernel<256, false>)<<<grid, 256, 0, s>>>(
            *cache, (int32_t)b0, k_items, v_items, k_ctas, dh, dk, dv, n_new, d_start_pos, sp_offset, k16, v16,
            d_err_flag);
        break;
    }
    const kvq_status ls = launch_status();
    if (ls != KVQ_OK) return ls;
  }
  return KVQ_OK;
}

}  // namespace kvq

extern "C" kvq_status kvq_append(const kvq_cache* cache, int32_t batch, int32_t n_new, const int32_t* d_start_pos,
                                 const void* k, const void* v, int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 0 || n_new < 0) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (batch == 0 || n_new == 0) return KVQ_OK;
  if (d_start_pos == nullptr || k == nullptr || v == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(k, 16) || !aligned_to(v, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* k16 = static_cast<const uint16_t*>(k);
  const uint16_t* v16 = static_cast<const uint16_t*>(v);
  if (is_fp4_layout(cache)) return launch_fp4_append(cache, batch, n_new, d_start_pos, 0, k16, v16, d_err_flag, s);
  const int64_t work = (int64_t)batch * n_new * cache->num_kv_heads * (cache->head_dim / 16);
  append_fp8_kernel<<<grid_for(work, 256), 256, 0, s>>>(*cache, batch, n_new, d_start_pos, k16, v16, d_err_flag);
  return launch_status();
}

extern "C" kvq_status kvq_fp8_set_scales(const kvq_cache* cache, int32_t batch, int32_t n, const void* k,
                                         const void* v, int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 0 || n < 0) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (cache->format != KVQ_FORMAT_FP8_E4M3_HEAD && cache->format != KVQ_FORMAT_NVFP4) return KVQ_ERR_INVALID_ARGUMENT;
  const float divisor = cache->format == KVQ_FORMAT_NVFP4 ? 2688.0f : 448.0f;  // 6 * 448 for NVFP4
  if ((int64_t)batch * n > 0 && (k == nullptr || v == nullptr)) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(k, 16) || !aligned_to(v, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  dim3 grid(cache->num_kv_heads, 2);
  fp8_scales_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      *cache, (int64_t)batch * n, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), divisor,
      d_err_flag);
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
