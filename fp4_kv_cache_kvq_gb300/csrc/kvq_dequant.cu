// kvq_dequant.cu -- expand a cache to dense fp32 or bf16 values.
//
// FP4: value = E2M1(code) * E4M3(scale) ("Quantising the KV cache", section
// "Code": the stored value is the rounded code times its block scale), read
// from the page pool's group layout (K by token, V by interleaved token pair).  The
// product has at most 6 significant bits and lies in [2^-10, 2688], so it is
// exact in fp32, f16 and bf16.  FP8 window: value = fp32(E4M3(code) * s_h).
//
// One thread per 16-value block: 8 code bytes + 1 scale byte in, 64 B (fp32)
// or 32 B (bf16) out with 16-byte stores.
#include <cuda_bf16.h>

#include "kvq_common.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ void store16(void* out, int64_t elem, const float (&x)[16], int out_dtype) {
  if (out_dtype == 0) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + elem);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
      w[q] = *reinterpret_cast<const uint32_t*>(&p);
    }
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + elem);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

__global__ void __launch_bounds__(256) dequant_fp4_kernel(const kvq_cache c, int32_t batch,
                                                          const int32_t* __restrict__ lens, int32_t max_len,
                                                          int out_dtype, void* k_out, void* v_out,
                                                          int32_t* flag) {
  const int nblk = c.head_dim >> 4;
  const int Hkv = c.num_kv_heads;
  const int P = c.page_size;
  const int64_t total = (int64_t)batch * max_len * Hkv * nblk;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % nblk);
    int64_t r = i / nblk;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int pos = (int)(r % max_len);
    const int b = (int)(r / max_len);
    const int32_t len = __ldg(lens + b);
    float kx[16], vx[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) kx[q] = vx[q] = 0.0f;
    bool ok = pos < len;
    if (len < 0) {
      set_flag(flag, KVQ_FLAG_BAD_LENGTH);
      ok = false;
    }
    const Fp4Layout L(c.head_dim, c.page_size);
    const uint8_t* grp = nullptr;
    int ls = 0;
    if (ok) {
      const int pg = pos / P;
      const int64_t phys = pg >= c.max_pages_per_seq ? -1
                           : c.page_table ? (int64_t)__ldg(c.page_table + (int64_t)b * c.max_pages_per_seq + pg)
                                          : (int64_t)b * c.max_pages_per_seq + pg;
      if (phys < 0 || phys >= c.num_pages) {
        set_flag(flag, KVQ_FLAG_PAGE_OOB);
        ok = false;
      } else {
        const int64_t off = L.group(phys, Hkv, h, pos % P);
        if (KVQ_IN(off >= 0 && off + L.group_bytes <= c.num_pages * (int64_t)Hkv * P * (9 * c.head_dim / 8), flag)) {
          grp = static_cast<const uint8_t*>(c.data) + off;
          ls = (pos % P) % L.G;
        } else {
          ok = false;
        }
      }
    }
    if (ok) {
      // K: 8 code bytes (channels 2k, 2k+1 per byte) and the block's scale
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(grp + (int64_t)ls * (c.head_dim / 2) + 8 * j));
      const float sk = e4m3_to_f32(__ldg(grp + L.k_scales() + (int64_t)ls * nblk + j));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float2 f = f16x2_to_float2(f16x2_from_e2m1x2(((q < 4 ? w.x : w.y) >> (8 * (q & 3))) & 0xFFu));
        kx[2 * q] = f.x * sk;
        kx[2 * q + 1] = f.y * sk;
      }
      // V: 16 interleaved bytes of the token pair; this token's nibbles
      const uint4 vw = __ldg(reinterpret_cast<const uint4*>(grp + L.v_block(ls >> 1, j)));
      const float sv = e4m3_to_f32(__ldg(grp + L.v_scale(ls, j)));
      const uint32_t ws[4] = {vw.x, vw.y, vw.z, vw.w};
      const int sh = 4 * (ls & 1);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t b0 = (ws[q >> 1] >> (16 * (q & 1) + sh)) & 0xFu;
        const uint32_t b1 = (ws[q >> 1] >> (16 * (q & 1) + 8 + sh)) & 0xFu;
        const float2 f = f16x2_to_float2(f16x2_from_e2m1x2(b0 | (b1 << 4)));
        vx[2 * q] = f.x * sv;
        vx[2 * q + 1] = f.y * sv;
      }
      if (c.format == KVQ_FORMAT_NVFP4) {  // second-level scales: fp32(value * S)
        const float Sk = __ldg(static_cast<const float*>(c.k_scale) + h);
        const float Sv = __ldg(static_cast<const float*>(c.v_scale) + h);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          kx[q] *= Sk;
          vx[q] *= Sv;
        }
      }
    }
    store16(k_out, i * 16, kx, out_dtype);
    store16(v_out, i * 16, vx, out_dtype);
  }
}

__global__ void __launch_bounds__(256) dequant_fp8_kernel(const kvq_cache c, int32_t batch, int out_dtype,
                                                          void* k_out, void* v_out) {
  const int nblk = c.head_dim >> 4;
  const int Hkv = c.num_kv_heads;
  const int W = c.page_size;
  const int64_t total = (int64_t)batch * W * Hkv * nblk;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % nblk);
    int64_t r = i / nblk;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int slot = (int)(r % W);
    const int b = (int)(r / W);
    const int64_t src = (((int64_t)b * Hkv + h) * W + slot) * c.head_dim + 16 * j;
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(side ? c.v_data : c.data) + src));
      const float s = __ldg(static_cast<const float*>(side ? c.v_scale : c.k_scale) + h);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      float x[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t two = (ws[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
        const float2 f = f16x2_to_float2(f16x2_from_e4m3x2(two));
        x[2 * q] = f.x * s;
        x[2 * q + 1] = f.y * s;
      }
      store16(side ? v_out : k_out, i * 16, x, out_dtype);
    }
  }
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_dequant(const kvq_cache* cache, int32_t batch, const int32_t* d_seq_lens, int32_t max_len,
                                  int32_t out_dtype, void* k_out, void* v_out, int32_t* d_err_flag,
                                  kvq_stream stream) {
  if (batch < 0 || max_len < 0 || (out_dtype != 0 && out_dtype != 1)) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (batch == 0 || max_len == 0) return KVQ_OK;
  if (k_out == nullptr || v_out == nullptr || !aligned_to(k_out, 16) || !aligned_to(v_out, 16))
    return KVQ_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t work = (int64_t)batch * max_len * cache->num_kv_heads * (cache->head_dim / 16);
  if (is_fp4_layout(cache)) {
    if (d_seq_lens == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    dequant_fp4_kernel<<<grid_for(work, 256), 256, 0, s>>>(*cache, batch, d_seq_lens, max_len, out_dtype, k_out,
                                                           v_out, d_err_flag);
  } else {
    if (max_len != cache->page_size) return KVQ_ERR_INVALID_ARGUMENT;
    dequant_fp8_kernel<<<grid_for(work, 256), 256, 0, s>>>(*cache, batch, out_dtype, k_out, v_out);
  }
  return launch_status();
}
