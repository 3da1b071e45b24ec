// kvq_decode.cuh -- pieces shared by the two decode kernels (the mma.sync
// kernel in kvq_decode.cu and the tcgen05 kernel in kvq_decode_tc.cu): the
// pool group geometry, the kernel parameters and the stream-K walk over the
// line of 128-token chunks of every (sequence, kv head) unit.
#pragma once

#include "kvq_common.cuh"

namespace kvq {

struct DecodeParams {
  const int32_t* lens;
  const int32_t* page_table;
  const uint8_t* pool;
  const uint16_t* q;
  float* part_o;
  float* part_ml;
  int2* unit_rec;
  int32_t* flag;
  const float* k_gscale;  // NVFP4 second-level scales [Hkv] (nullptr: plain FP4)
  const float* v_gscale;
  int64_t num_pages;
  int32_t batch, hkv, g, hq, page, max_pages, window, head_dim;
  float qk_log2;  // softmax_scale * log2(e)
  // fused append of each sequence's newest token (position T_b - 1) before
  // the decode reads it (kvq_append_decode_attn); k_new == nullptr: none
  const uint16_t* k_new;  // bf16 [batch][Hkv][head_dim]
  const uint16_t* v_new;
  kvq_cache cache;        // the FP4 / NVFP4 cache written
  int32_t nvfp4;
  uint64_t wait_ns;       // 0, or a test's shortened limit of the mma.sync kernel's work waits (ns)
  int64_t pool_bytes;     // bytes of the FP4 pool, and partial slots of the workspace (bounds checks)
  int64_t n_slots;
};

// The merge of the per-range partials (and of the FP8 window's terms).
struct MergeParams {
  const int32_t* lens;
  const uint16_t* q;
  const float* part_o;
  const float* part_ml;
  const int2* unit_rec;
  float* out;
  int32_t* flag;
  // FP8 window (k8 == nullptr: none)
  const uint8_t* k8;
  const uint8_t* v8;
  const float* k8_scale;
  const float* v8_scale;
  int32_t window;
  int32_t hkv, g, hq, head_dim;
  float qk_log2;
  int64_t n_slots;        // partial slots of the workspace, sequences (bounds checks)
  int32_t batch;
};

// The decode kernels: mma.sync (kvq_decode_kernel.cuh; head_dim 64 or 128,
// `ctas` persistent CTAs, three per SM), instantiated with the fixed wait
// limit (kvq_decode.cu) and with the limit dp.wait_ns (kvq_decode_test_wait.cu,
// launched only while a test has set one); and the head_dim 128 tcgen05
// variant (kvq_decode_tc.cu; one CTA per SM with three pipelines, i.e. the
// ranges and partial slots of 3 x (number of SMs) CTAs; fixed limit only).
// `after_append`: launch as a programmatic dependent of the append kernel
// enqueued just before (the producer waits for it before its first copy).
kvq_status launch_decode_mma(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append);
kvq_status launch_decode_mma_test_wait(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append);
kvq_status launch_decode_tc(const DecodeParams& dp, cudaStream_t s);
// The merge launch (kvq_merge.cu), a programmatic dependent of the decode
// launch just enqueued: merge_splits_kernel, or merge_window_kernel when
// mp.k8 is set.
kvq_status launch_merge(const MergeParams& mp, int64_t units, cudaStream_t s);

namespace {

constexpr int kChunk = 128;          // tokens per pipeline stage
constexpr int kNG = 8;  // query rows per kv head held by one tile (G <= 8)
constexpr float kLazySlack = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWindow = 1024;  // largest FP8 window the window merge takes

// Compile-time view of one pool group of GT tokens (see Fp4Layout).
template <int D, int GT>
struct Grp {
  static constexpr int kNB = D / 16;
  static constexpr int kBytes = GT * 9 * D / 8;
  static constexpr int kKS = GT * D / 2;          // K scales
  static constexpr int kVC = GT * (D / 2 + kNB);  // V codes (token pairs)
  static constexpr int kVS = GT * (D + kNB);      // V scales (token pairs)
};


__device__ __forceinline__ int fp4_chunks(int32_t T, int window) {
  if (T <= 0) return 0;
  const int w = window > 0 ? min(window, T) : 0;
  return (T - w + kChunk - 1) / kChunk;
}

__device__ __forceinline__ int fp4_tokens(int32_t T, int window) {
  if (T <= 0) return 0;
  const int w = window > 0 ? min(window, T) : 0;
  return T - w;
}

// Position of a walker on the line of chunks: unit (b, h), chunk c of nch.
struct Walker {
  int b, h, c, nch;
  int64_t v;  // index on the line
};

// Every warp computes the same thing: the line's length and where range
// `idx` of `count` equal ranges starts.  Lanes scan 32 sequences at a time.
__device__ __forceinline__ void plan(const DecodeParams& p, int idx, int count, int64_t& total, int64_t& v0,
                                     int64_t& v1, Walker& wk) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  total = 0;
  // pass 1: total
  for (int base = 0; base < p.batch; base += 32) {
    const int bb = base + lane;
    int64_t x = bb < p.batch ? (int64_t)fp4_chunks(__ldg(p.lens + bb), p.window) * p.hkv : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    acc += x;
  }
  total = acc;
  const int64_t per = (total + count - 1) / count;
  v0 = min(total, (int64_t)idx * per);
  v1 = min(total, v0 + per);
  wk.b = p.batch;
  wk.h = 0;
  wk.c = 0;
  wk.nch = 0;
  wk.v = v0;
  if (v0 >= v1) return;
  // pass 2: locate v0
  acc = 0;
  for (int base = 0; base < p.batch; base += 32) {
    const int bb = base + lane;
    const int n = bb < p.batch ? fp4_chunks(__ldg(p.lens + bb), p.window) : 0;
    const int64_t x = (int64_t)n * p.hkv;
    int64_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const int64_t group_total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (acc + group_total > v0) {
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, acc + incl > v0);
      const int L = __ffs(hit) - 1;
      const int64_t before = acc + __shfl_sync(0xFFFFFFFFu, incl - x, L);
      const int nL = __shfl_sync(0xFFFFFFFFu, n, L);
      const int64_t rem = v0 - before;
      wk.b = base + L;
      wk.nch = nL;
      wk.h = (int)(rem / nL);
      wk.c = (int)(rem % nL);
      return;
    }
    acc += group_total;
  }
}

__device__ __forceinline__ void advance(const DecodeParams& p, Walker& wk) {
  ++wk.v;
  if (++wk.c < wk.nch) return;
  wk.c = 0;
  if (++wk.h < p.hkv) return;
  wk.h = 0;
  do {
    ++wk.b;
    wk.nch = wk.b < p.batch ? fp4_chunks(__ldg(p.lens + wk.b), p.window) : 1;
  } while (wk.nch == 0);
}

}  // namespace
}  // namespace kvq
