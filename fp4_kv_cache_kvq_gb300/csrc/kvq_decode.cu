// kvq_decode.cu -- split-K flash-decode attention over the FP4 paged cache,
// plus the merge kernel that folds in the FP8 sliding window and combines the
// splits.
//
// Method: "Quantising the KV cache", section "Code" -- the quantised K and V
// feed an otherwise unchanged attention, out = softmax(scale * q.K^T) V^.
// "Quantising the KV cache", section "Concept" and "KV Cache Quantisation",
// section "Common questions": decode is a stream over the whole cache, and the
// saving only holds if the kernel does the scale handling and dequantisation
// itself -- here codes and scales are read once from HBM and expanded in
// registers right before the tensor-core products.
//
// Work decomposition (stream-K over the whole batch).  Every (sequence b,
// kv head h) pair is a unit; its FP4 positions are cut into chunks of 64
// tokens.  All units' chunks are laid end to end and the persistent grid (two
// CTAs per SM) splits that line into equal contiguous ranges, so ragged
// lengths balance to within one chunk.  A CTA writes one partial (m, l, o) per
// unit it touches; the merge kernel combines them.
//
// CTA = 4 consumer warps + 1 producer warp.  The producer's lane 0 streams the
// chunk's K codes and V codes (3-D tiled TMA loads, 64-byte swizzle for
// head_dim 128) and K/V scale bytes (1-D bulk copies) into an 8-stage ring
// guarded by mbarriers.  Consumer warp w takes tokens [16w, 16w+16) of each
// chunk and runs, per 16 tokens:
//   S^T(16 tok x 8 q-rows) = K^(16 x d) Q^T    mma.m16n8k16, K^ dequantised in
//                                              registers (cvt e2m1x2->f16x2,
//                                              times the block scale)
//   online softmax in the log2 domain with lazy rescaling (the running max is
//   only raised when a score exceeds it by more than 8)
//   O^T(d x 8) += V^T(d x 16 tok) P^T           mma.m16n8k16, P in f16
// Tokens sit on the MMA's M side so a GQA group of up to 8 query heads fills
// N = 8 without padding rows.  The query is pre-scaled per head by a power of
// two so that its bf16 values are exact in f16; the factor is undone in fp32.
#include "kvq_common.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {

constexpr int kChunk = 64;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStages = 8;
constexpr int kNG = 8;  // query rows per kv head held by one tile (G <= 8)
constexpr float kLazySlack = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWindow = 1024;

template <int D>
struct Geo {
  static constexpr int kCodeRow = D / 2;
  static constexpr int kScaleRow = D / 16;
  static constexpr int kCodeBytes = kChunk * kCodeRow;
  static constexpr int kScaleBytes = kChunk * kScaleRow;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kCodeBytes;
  static constexpr int kOffKS = 2 * kCodeBytes;
  static constexpr int kOffVS = 2 * kCodeBytes + kScaleBytes;
  static constexpr int kStageBytes = ((2 * kCodeBytes + 2 * kScaleBytes) + 1023) / 1024 * 1024;
  // flush buffer: O[warp][row][D], M[warp][row], L[warp][row]
  static constexpr int kFlushBytes = kConsumerWarps * kNG * (D + 2) * 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + kFlushBytes + 2 * kStages * 8 + kStages * 4 + 16 + 1024;
};

struct DecodeParams {
  const int32_t* lens;
  const int32_t* page_table;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint16_t* q;
  float* part_o;
  float* part_ml;
  int2* unit_rec;
  int32_t* flag;
  int64_t num_pages;
  int32_t batch, hkv, g, hq, page, max_pages, window;
  float qk_log2;  // softmax_scale * log2(e)
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

// Every warp computes the same thing: the line's length and where this CTA's
// range starts.  Lanes scan 32 sequences at a time.
__device__ __forceinline__ void plan(const DecodeParams& p, int64_t& total, int64_t& v0, int64_t& v1, Walker& wk) {
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
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  v0 = min(total, (int64_t)blockIdx.x * per);
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

// Shared-memory carve-up.
template <int D>
struct Smem {
  uint8_t* stages;
  float* flush_o;  // [warp][row][D]
  float* flush_m;  // [warp][row]
  float* flush_l;  // [warp][row]
  uint64_t* full;
  uint64_t* empty;
  int* ntok;
  int* abort;
};

template <int D>
__device__ __forceinline__ Smem<D> carve(uint8_t* raw) {
  using G = Geo<D>;
  Smem<D> s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stages = base;
  uint8_t* ptr = base + kStages * G::kStageBytes;
  s.flush_o = reinterpret_cast<float*>(ptr);
  ptr += kConsumerWarps * kNG * D * 4;
  s.flush_m = reinterpret_cast<float*>(ptr);
  ptr += kConsumerWarps * kNG * 4;
  s.flush_l = reinterpret_cast<float*>(ptr);
  ptr += kConsumerWarps * kNG * 4;
  s.full = reinterpret_cast<uint64_t*>(ptr);
  ptr += kStages * 8;
  s.empty = reinterpret_cast<uint64_t*>(ptr);
  ptr += kStages * 8;
  s.ntok = reinterpret_cast<int*>(ptr);
  ptr += kStages * 4;
  s.abort = reinterpret_cast<int*>(ptr);
  return s;
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void producer(const DecodeParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv, Smem<D>& sm,
                         Walker wk, int64_t v1) {
  using G = Geo<D>;
  const int P = p.page;
  const int rows_per_copy = P < kChunk ? P : kChunk;
  uint32_t it = 0;
  for (; wk.v < v1; advance(p, wk), ++it) {
    const uint32_t s = it % kStages;
    if (it >= (uint32_t)kStages) {
      if (!mbar_wait(smem_addr(&sm.empty[s]), ((it / kStages) + 1) & 1)) {
        set_flag(p.flag, KVQ_FLAG_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort) = 1;
        break;
      }
    }
    if (*reinterpret_cast<volatile int*>(sm.abort)) break;
    const int n4 = fp4_tokens(__ldg(p.lens + wk.b), p.window);
    const int tok0 = wk.c * kChunk;
    const int ntok = min(kChunk, n4 - tok0);
    const int ncopies = P < kChunk ? (ntok + P - 1) / P : 1;
    const int pg0 = tok0 / P;
    const int off0 = P < kChunk ? 0 : tok0 % P;
    int64_t phys[kChunk / 16];
    bool ok = true;
    for (int i = 0; i < ncopies; ++i) {
      const int pg = pg0 + i;
      int64_t ph = -1;
      if (pg < p.max_pages)
        ph = p.page_table ? (int64_t)__ldg(p.page_table + (int64_t)wk.b * p.max_pages + pg)
                          : (int64_t)wk.b * p.max_pages + pg;
      if (ph < 0 || ph >= p.num_pages) ok = false;
      phys[i] = ph;
    }
    const uint32_t full = smem_addr(&sm.full[s]);
    uint8_t* st = sm.stages + s * G::kStageBytes;
    if (!ok) {
      set_flag(p.flag, KVQ_FLAG_PAGE_OOB);
      sm.ntok[s] = 0;
      mbar_arrive(full);
      continue;
    }
    sm.ntok[s] = ntok;
    const uint32_t code_bytes = (uint32_t)(ncopies * rows_per_copy * G::kCodeRow);
    const uint32_t scale_bytes = (uint32_t)(ncopies * rows_per_copy * G::kScaleRow);
    mbar_arrive_expect_tx(full, 2 * code_bytes + 2 * scale_bytes);
    for (int i = 0; i < ncopies; ++i) {
      const int64_t row0 = (phys[i] * p.hkv + wk.h) * P + off0;  // token row in the pool
      const int z = (int)(phys[i] * p.hkv + wk.h);
      const uint32_t dk = smem_addr(st + G::kOffK + i * rows_per_copy * G::kCodeRow);
      const uint32_t dv = smem_addr(st + G::kOffV + i * rows_per_copy * G::kCodeRow);
      tma_load_3d(dk, tmk, 0, off0, z, full);
      tma_load_3d(dv, tmv, 0, off0, z, full);
      bulk_g2s(smem_addr(st + G::kOffKS + i * rows_per_copy * G::kScaleRow), p.k_scales + row0 * G::kScaleRow,
               rows_per_copy * G::kScaleRow, full);
      bulk_g2s(smem_addr(st + G::kOffVS + i * rows_per_copy * G::kScaleRow), p.v_scales + row0 * G::kScaleRow,
               rows_per_copy * G::kScaleRow, full);
    }
  }
  // Wait for every copy still in flight before the CTA can retire.
  const uint32_t issued = it;
  const uint32_t first = issued > (uint32_t)kStages ? issued - kStages : 0;
  for (uint32_t j = first; j < issued; ++j) {
    if (!mbar_wait(smem_addr(&sm.full[j % kStages]), (j / kStages) & 1)) {
      set_flag(p.flag, KVQ_FLAG_TIMEOUT);
      break;
    }
  }
}

// ------------------------------------------------------------------ consumer
template <int D>
struct ConsumerState {
  float o[D / 16][4];
  uint32_t qf[D / 8];
  float cs[2];
  float m[2];
  float l[2];
};

template <int D>
__device__ __forceinline__ void begin_unit(const DecodeParams& p, ConsumerState<D>& st, int b, int h) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  constexpr int kPer = D / 4;  // channels of q per thread
  float v[kPer];
  float amax = 0.0f;
  if (g < p.g) {
    const uint16_t* src = p.q + ((int64_t)b * p.hq + (int64_t)h * p.g + g) * D + tig * kPer;
#pragma unroll
    for (int i = 0; i < kPer / 8; ++i) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + i);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[8 * i + 2 * k] = bf16_lo(ws[k]);
        v[8 * i + 2 * k + 1] = bf16_hi(ws[k]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = 0.0f;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  // power-of-two prescale: max |q| * 2^k in [2^14, 2^15) keeps bf16 values exact in f16
  int k = 0;
  if (amax > 0.0f && amax <= 3.4e38f) {
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
    k = min(100, max(-113, 14 - e));
  }
  const float up = __uint_as_float((uint32_t)(k + 127) << 23);
#pragma unroll
  for (int i = 0; i < D / 8; ++i) st.qf[i] = pack_f16x2(v[2 * i] * up, v[2 * i + 1] * up);
  const int k0 = __shfl_sync(0xFFFFFFFFu, k, (2 * tig) * 4);
  const int k1 = __shfl_sync(0xFFFFFFFFu, k, (2 * tig + 1) * 4);
  st.cs[0] = p.qk_log2 * __uint_as_float((uint32_t)(127 - k0) << 23);
  st.cs[1] = p.qk_log2 * __uint_as_float((uint32_t)(127 - k1) << 23);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mt][i] = 0.0f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.0f;
}

// Broadcast a K scale byte into both halves of an f16x2.
__device__ __forceinline__ uint32_t scale_pair_same(uint32_t byte) { return f16x2_from_e4m3x2(byte * 0x0101u); }

template <int D>
__device__ __forceinline__ void process_slice(const DecodeParams& p, ConsumerState<D>& st, const uint8_t* stage,
                                              int ntok, uint32_t empty_bar) {
  using G = Geo<D>;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int r0 = 16 * warp;
  const uint8_t* sK = stage + G::kOffK;
  const uint8_t* sV = stage + G::kOffV;
  const uint8_t* sKS = stage + G::kOffKS;
  const uint8_t* sVS = stage + G::kOffVS;
  // V k-slot order: pair A = tokens (tA, tA+8), pair B = (tB, tB+8); the
  // parity flip keeps the 8-byte V loads of a half-warp on distinct banks.
  const int tA = 2 * tig + (tig & 1);
  const int tB = 2 * tig + 1 - (tig & 1);
  const int rowK0 = r0 + g, rowK1 = r0 + g + 8;
  const int rVA0 = r0 + tA, rVA1 = r0 + tA + 8, rVB0 = r0 + tB, rVB1 = r0 + tB + 8;

  // ---- loads from the stage (then release it)
  uint32_t kw0[D / 32], kw1[D / 32];  // the thread's D/16 code bytes of rows g, g+8
  uint32_t ksA, ksB;                  // K scale bytes (D=128: 2 per row, D=64: 1 per row)
  uint32_t vA0[D / 64], vA1[D / 64], vB0[D / 64], vB1[D / 64];
  uint32_t vsA, vsB;
  if constexpr (D == 128) {
    const int gr = tig ^ ((rowK0 >> 1) & 3);
    const uint4 a = *reinterpret_cast<const uint4*>(sK + rowK0 * 64 + gr * 16);
    const uint4 b = *reinterpret_cast<const uint4*>(sK + rowK1 * 64 + gr * 16);
    kw0[0] = a.x; kw0[1] = a.y; kw0[2] = a.z; kw0[3] = a.w;
    kw1[0] = b.x; kw1[1] = b.y; kw1[2] = b.z; kw1[3] = b.w;
    ksA = *reinterpret_cast<const uint16_t*>(sKS + rowK0 * 8 + 2 * tig);
    ksB = *reinterpret_cast<const uint16_t*>(sKS + rowK1 * 8 + 2 * tig);
    const int vo = 8 * (g & 1);
    const uint2 a0 = *reinterpret_cast<const uint2*>(sV + rVA0 * 64 + (((g >> 1) ^ ((rVA0 >> 1) & 3)) * 16) + vo);
    const uint2 a1 = *reinterpret_cast<const uint2*>(sV + rVA1 * 64 + (((g >> 1) ^ ((rVA1 >> 1) & 3)) * 16) + vo);
    const uint2 b0 = *reinterpret_cast<const uint2*>(sV + rVB0 * 64 + (((g >> 1) ^ ((rVB0 >> 1) & 3)) * 16) + vo);
    const uint2 b1 = *reinterpret_cast<const uint2*>(sV + rVB1 * 64 + (((g >> 1) ^ ((rVB1 >> 1) & 3)) * 16) + vo);
    vA0[0] = a0.x; vA0[1] = a0.y; vA1[0] = a1.x; vA1[1] = a1.y;
    vB0[0] = b0.x; vB0[1] = b0.y; vB1[0] = b1.x; vB1[1] = b1.y;
    vsA = sVS[rVA0 * 8 + g] | (sVS[rVA1 * 8 + g] << 8);
    vsB = sVS[rVB0 * 8 + g] | (sVS[rVB1 * 8 + g] << 8);
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(sK + rowK0 * 32 + 8 * tig);
    const uint2 b = *reinterpret_cast<const uint2*>(sK + rowK1 * 32 + 8 * tig);
    kw0[0] = a.x; kw0[1] = a.y;
    kw1[0] = b.x; kw1[1] = b.y;
    ksA = sKS[rowK0 * 4 + tig];
    ksB = sKS[rowK1 * 4 + tig];
    vA0[0] = *reinterpret_cast<const uint32_t*>(sV + rVA0 * 32 + 4 * g);
    vA1[0] = *reinterpret_cast<const uint32_t*>(sV + rVA1 * 32 + 4 * g);
    vB0[0] = *reinterpret_cast<const uint32_t*>(sV + rVB0 * 32 + 4 * g);
    vB1[0] = *reinterpret_cast<const uint32_t*>(sV + rVB1 * 32 + 4 * g);
    vsA = sVS[rVA0 * 4 + (g >> 1)] | (sVS[rVA1 * 4 + (g >> 1)] << 8);
    vsB = sVS[rVB0 * 4 + (g >> 1)] | (sVS[rVB1 * 4 + (g >> 1)] << 8);
  }
  mbar_arrive(empty_bar);

  // ---- S^T = K^ Q^T  (rows: tokens g, g+8; cols: q rows)
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  uint32_t sA0, sA1, sB0, sB1;
  if constexpr (D == 128) {
    sA0 = scale_pair_same(ksA & 0xFFu);
    sA1 = scale_pair_same(ksA >> 8);
    sB0 = scale_pair_same(ksB & 0xFFu);
    sB1 = scale_pair_same(ksB >> 8);
  } else {
    sA0 = sA1 = scale_pair_same(ksA);
    sB0 = sB1 = scale_pair_same(ksB);
  }
#pragma unroll
  for (int j = 0; j < D / 16; ++j) {
    const int sh = 16 * (j & 1);
    const uint32_t wA = kw0[j >> 1], wB = kw1[j >> 1];
    const uint32_t scA = (D == 128 && j >= 4) ? sA1 : sA0;
    const uint32_t scB = (D == 128 && j >= 4) ? sB1 : sB0;
    const uint32_t a0 = hmul2_u32(f16x2_from_e2m1x2(wA >> sh), scA);
    const uint32_t a1 = hmul2_u32(f16x2_from_e2m1x2(wB >> sh), scB);
    const uint32_t a2 = hmul2_u32(f16x2_from_e2m1x2(wA >> (sh + 8)), scA);
    const uint32_t a3 = hmul2_u32(f16x2_from_e2m1x2(wB >> (sh + 8)), scB);
    mma_f16_16816(acc[j & 1], a0, a1, a2, a3, st.qf[2 * j], st.qf[2 * j + 1]);
  }
  float x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = (acc[0][i] + acc[1][i]) * st.cs[i & 1];
  if (r0 + g >= ntok) x[0] = x[1] = -INFINITY;
  if (r0 + g + 8 >= ntok) x[2] = x[3] = -INFINITY;

  // ---- online softmax (log2 domain, lazy rescale)
  const bool need = fmaxf(x[0], x[2]) > st.m[0] + kLazySlack || fmaxf(x[1], x[3]) > st.m[1] + kLazySlack;
  if (__any_sync(0xFFFFFFFFu, need)) {
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
    }
    const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
    const float al0 = (st.m[0] == -INFINITY) ? 0.0f : fast_exp2(st.m[0] - n0);
    const float al1 = (st.m[1] == -INFINITY) ? 0.0f : fast_exp2(st.m[1] - n1);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.o[mt][0] *= al0;
      st.o[mt][2] *= al0;
      st.o[mt][1] *= al1;
      st.o[mt][3] *= al1;
    }
    st.l[0] *= al0;
    st.l[1] *= al1;
    st.m[0] = n0;
    st.m[1] = n1;
  }
  const float ref0 = st.m[0] == -INFINITY ? 0.0f : st.m[0];
  const float ref1 = st.m[1] == -INFINITY ? 0.0f : st.m[1];
  const float p0 = fast_exp2(x[0] - ref0), p2 = fast_exp2(x[2] - ref0);
  const float p1 = fast_exp2(x[1] - ref1), p3 = fast_exp2(x[3] - ref1);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  const uint32_t xp = pack_f16x2(p0, p2);  // q row 2tig: tokens (g, g+8)
  const uint32_t yp = pack_f16x2(p1, p3);  // q row 2tig+1
  const int srcA = 4 * tA + (g >> 1), srcB = 4 * tB + (g >> 1);
  const uint32_t XA = __shfl_sync(0xFFFFFFFFu, xp, srcA), YA = __shfl_sync(0xFFFFFFFFu, yp, srcA);
  const uint32_t XB = __shfl_sync(0xFFFFFFFFu, xp, srcB), YB = __shfl_sync(0xFFFFFFFFu, yp, srcB);
  const uint32_t pbA = (g & 1) ? YA : XA;
  const uint32_t pbB = (g & 1) ? YB : XB;

  // ---- O^T += V^T P^T
  // masked tokens get a zero V scale so stale bytes cannot inject NaN
  if (r0 + tA >= ntok) vsA &= 0xFF00u;
  if (r0 + tA + 8 >= ntok) vsA &= 0x00FFu;
  if (r0 + tB >= ntok) vsB &= 0xFF00u;
  if (r0 + tB + 8 >= ntok) vsB &= 0x00FFu;
  const uint32_t svA = f16x2_from_e4m3x2(vsA);
  const uint32_t svB = f16x2_from_e4m3x2(vsB);
  if constexpr (D == 128) {
    uint32_t lo[2][2], hi[2][2];  // [pair A/B][x (ch 0-7) / y (ch 8-15)]
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      lo[0][q] = (vA0[q] & 0x0F0F0F0Fu) | ((vA1[q] & 0x0F0F0F0Fu) << 4);
      hi[0][q] = ((vA0[q] >> 4) & 0x0F0F0F0Fu) | (vA1[q] & 0xF0F0F0F0u);
      lo[1][q] = (vB0[q] & 0x0F0F0F0Fu) | ((vB1[q] & 0x0F0F0F0Fu) << 4);
      hi[1][q] = ((vB0[q] >> 4) & 0x0F0F0F0Fu) | (vB1[q] & 0xF0F0F0F0u);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int sh = 8 * (mt >> 1);
      const uint32_t a0 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hi[0][0] : lo[0][0]) >> sh), svA);
      const uint32_t a1 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hi[0][1] : lo[0][1]) >> sh), svA);
      const uint32_t a2 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hi[1][0] : lo[1][0]) >> sh), svB);
      const uint32_t a3 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hi[1][1] : lo[1][1]) >> sh), svB);
      mma_f16_16816(st.o[mt], a0, a1, a2, a3, pbA, pbB);
    }
  } else {
    const uint32_t loA = (vA0[0] & 0x0F0F0F0Fu) | ((vA1[0] & 0x0F0F0F0Fu) << 4);
    const uint32_t hiA = ((vA0[0] >> 4) & 0x0F0F0F0Fu) | (vA1[0] & 0xF0F0F0F0u);
    const uint32_t loB = (vB0[0] & 0x0F0F0F0Fu) | ((vB1[0] & 0x0F0F0F0Fu) << 4);
    const uint32_t hiB = ((vB0[0] >> 4) & 0x0F0F0F0Fu) | (vB1[0] & 0xF0F0F0F0u);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int sh0 = 8 * (mt >> 1), sh1 = 8 * (2 + (mt >> 1));
      const uint32_t a0 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hiA : loA) >> sh0), svA);
      const uint32_t a1 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hiA : loA) >> sh1), svA);
      const uint32_t a2 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hiB : loB) >> sh0), svB);
      const uint32_t a3 = hmul2_u32(f16x2_from_e2m1x2(((mt & 1) ? hiB : loB) >> sh1), svB);
      mma_f16_16816(st.o[mt], a0, a1, a2, a3, pbA, pbB);
    }
  }
}

// Combine the four warps' states for one unit and write the CTA's partial.
template <int D>
__device__ void flush_unit(const DecodeParams& p, ConsumerState<D>& st, Smem<D>& sm, int64_t slot) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l[0] += __shfl_xor_sync(0xFFFFFFFFu, st.l[0], o);
    st.l[1] += __shfl_xor_sync(0xFFFFFFFFu, st.l[1], o);
  }
  named_barrier_sync(1, 32 * kConsumerWarps);
  float* ow = sm.flush_o + warp * kNG * D;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int c0 = (D / 8) * g + mt, c1 = (D / 8) * g + D / 16 + mt;
    ow[(2 * tig) * D + c0] = st.o[mt][0];
    ow[(2 * tig + 1) * D + c0] = st.o[mt][1];
    ow[(2 * tig) * D + c1] = st.o[mt][2];
    ow[(2 * tig + 1) * D + c1] = st.o[mt][3];
  }
  if (g == 0) {
    sm.flush_m[warp * kNG + 2 * tig] = st.m[0];
    sm.flush_m[warp * kNG + 2 * tig + 1] = st.m[1];
    sm.flush_l[warp * kNG + 2 * tig] = st.l[0];
    sm.flush_l[warp * kNG + 2 * tig + 1] = st.l[1];
  }
  named_barrier_sync(1, 32 * kConsumerWarps);
  for (int idx = tid; idx < p.g * D; idx += 32 * kConsumerWarps) {
    const int r = idx / D, ch = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm.flush_m[w * kNG + r]);
    float o = 0.0f, l = 0.0f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = sm.flush_m[w * kNG + r];
        const float f = mw == -INFINITY ? 0.0f : fast_exp2(mw - mx);
        o += f * sm.flush_o[(w * kNG + r) * D + ch];
        l += f * sm.flush_l[w * kNG + r];
      }
    }
    p.part_o[(slot * p.g + r) * D + ch] = o;
    if (ch == 0) {
      p.part_ml[(slot * p.g + r) * 2 + 0] = mx;
      p.part_ml[(slot * p.g + r) * 2 + 1] = l;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    decode_fp4_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const DecodeParams p) {
  using G = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem<D> sm = carve<D>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), 32 * kConsumerWarps);
    }
    *sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  int64_t total, v0, v1;
  Walker wk;
  plan(p, total, v0, v1, wk);
  if (v0 >= v1) return;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      producer<D>(p, &tmk, &tmv, sm, wk, v1);
    }
    return;
  }

  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  ConsumerState<D> st;
  bool have = false, dead = false;
  int64_t slot = 0;
  uint32_t it = 0;
  for (; wk.v < v1; advance(p, wk), ++it) {
    if (!have || wk.c == 0) {
      if (have) flush_unit<D>(p, st, sm, slot);
      const int64_t u = (int64_t)wk.b * p.hkv + wk.h;
      slot = u + blockIdx.x;
      begin_unit<D>(p, st, wk.b, wk.h);
      have = true;
      if (wk.c == 0 && threadIdx.x == 0) {
        const int64_t last_cta = (wk.v + wk.nch - 1) / per;
        p.unit_rec[u] = make_int2((int)slot, (int)(last_cta - blockIdx.x + 1));
      }
    }
    if (dead) continue;
    const uint32_t s = it % kStages;
    bool ok = !*reinterpret_cast<volatile int*>(sm.abort) && mbar_wait(smem_addr(&sm.full[s]), (it / kStages) & 1);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (!ok) {
      dead = true;
      if (lane == 0) {
        set_flag(p.flag, KVQ_FLAG_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort) = 1;
      }
      continue;
    }
    const int ntok = sm.ntok[s];
    if (ntok > 16 * warp) {
      process_slice<D>(p, st, sm.stages + s * G::kStageBytes, ntok, smem_addr(&sm.empty[s]));
    } else {
      mbar_arrive(smem_addr(&sm.empty[s]));
    }
  }
  if (have) flush_unit<D>(p, st, sm, slot);
}

// ------------------------------------------------------------------ merge (+ FP8 window)
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
};

// One CTA per unit (b, kv head): FP8 window attention for the unit's query
// rows (fp32 products x^ = E4M3(c) * s_h, fp32 dot products), then the
// log-sum-exp merge of that window with every FP4 partial of the unit.
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  extern __shared__ float msm[];
  const int D = p.head_dim;
  const int u = blockIdx.x;
  const int b = u / p.hkv, h = u % p.hkv;
  const int tid = threadIdx.x;
  int32_t T = __ldg(p.lens + b);
  if (T < 0) {
    if (tid == 0 && h == 0) set_flag(p.flag, KVQ_FLAG_BAD_LENGTH);
    T = 0;
  }
  const int w = (p.k8 != nullptr) ? min(p.window, T) : 0;
  const int nch = (T - w + kChunk - 1) / kChunk;
  float* qs = msm;                       // [G][D]
  float* sc = qs + kNG * D;              // [G][window]
  float* mw = sc + kNG * max(p.window, 1);  // [G] window max
  float* lw = mw + kNG;                  // [G] window sum
  float* ow = lw + kNG;                  // [G][D] window numerator
  if (w > 0) {
    for (int i = tid; i < p.g * D; i += blockDim.x) {
      const int r = i / D, ch = i % D;
      const uint16_t bits = p.q[((int64_t)b * p.hq + (int64_t)h * p.g + r) * D + ch];
      qs[i] = __uint_as_float((uint32_t)bits << 16);
    }
    __syncthreads();
    const float sk = __ldg(p.k8_scale + h), sv = __ldg(p.v8_scale + h);
    for (int t = tid; t < w; t += blockDim.x) {
      const int pos = T - w + t;
      const uint8_t* krow = p.k8 + (((int64_t)b * p.hkv + h) * p.window + (pos % p.window)) * D;
      float acc[kNG];
#pragma unroll
      for (int r = 0; r < kNG; ++r) acc[r] = 0.0f;
      for (int ch = 0; ch < D; ch += 16) {
        const uint4 cw = *reinterpret_cast<const uint4*>(krow + ch);
        const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float2 f = f16x2_to_float2(f16x2_from_e4m3x2((ws[q >> 1] >> (16 * (q & 1))) & 0xFFFFu));
          const float x0 = f.x * sk, x1 = f.y * sk;
#pragma unroll
          for (int r = 0; r < kNG; ++r) {
            if (r < p.g) {
              acc[r] = fmaf(qs[r * D + ch + 2 * q], x0, acc[r]);
              acc[r] = fmaf(qs[r * D + ch + 2 * q + 1], x1, acc[r]);
            }
          }
        }
      }
      for (int r = 0; r < p.g; ++r) sc[r * p.window + t] = acc[r] * p.qk_log2;
    }
    __syncthreads();
    // per q row: max, then weights in place, then the sum
    const int warp = tid >> 5, lane = tid & 31;
    for (int r = warp; r < p.g; r += 4) {
      float mx = -INFINITY;
      for (int t = lane; t < w; t += 32) mx = fmaxf(mx, sc[r * p.window + t]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      float l = 0.0f;
      for (int t = lane; t < w; t += 32) {
        const float e = fast_exp2(sc[r * p.window + t] - mx);
        sc[r * p.window + t] = e;
        l += e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
      if (lane == 0) {
        mw[r] = mx;
        lw[r] = l;
      }
    }
    __syncthreads();
    for (int i = tid; i < p.g * D; i += blockDim.x) {
      const int r = i / D, ch = i % D;
      float o = 0.0f;
      for (int t = 0; t < w; ++t) {
        const int pos = T - w + t;
        const uint8_t c = p.v8[(((int64_t)b * p.hkv + h) * p.window + (pos % p.window)) * D + ch];
        const float x = e4m3_to_f32(c) * sv;
        o = fmaf(sc[r * p.window + t], x, o);
      }
      ow[i] = o;
    }
    __syncthreads();
  }
  int2 rec = make_int2(0, 0);
  if (nch > 0) rec = p.unit_rec[u];
  for (int i = tid; i < p.g * D; i += blockDim.x) {
    const int r = i / D, ch = i % D;
    float mx = w > 0 ? mw[r] : -INFINITY;
    for (int k = 0; k < rec.y; ++k) mx = fmaxf(mx, p.part_ml[((int64_t)(rec.x + k) * p.g + r) * 2]);
    float o = 0.0f, l = 0.0f;
    if (mx != -INFINITY) {
      if (w > 0) {
        const float f = mw[r] == -INFINITY ? 0.0f : fast_exp2(mw[r] - mx);
        o += f * ow[i];
        l += f * lw[r];
      }
      for (int k = 0; k < rec.y; ++k) {
        const int64_t sl = rec.x + k;
        const float m = p.part_ml[(sl * p.g + r) * 2];
        const float f = m == -INFINITY ? 0.0f : fast_exp2(m - mx);
        o += f * p.part_o[(sl * p.g + r) * D + ch];
        l += f * p.part_ml[(sl * p.g + r) * 2 + 1];
      }
    }
    p.out[((int64_t)b * p.hq + (int64_t)h * p.g + r) * D + ch] = l > 0.0f ? o / l : 0.0f;
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<EncodeTiledFn>(fn);
}

bool make_code_map(EncodeTiledFn enc, CUtensorMap* map, void* base, const kvq_cache& c) {
  const cuuint64_t row = (cuuint64_t)c.head_dim / 2;
  cuuint64_t dims[3] = {row, (cuuint64_t)c.page_size, (cuuint64_t)c.num_pages * (cuuint64_t)c.num_kv_heads};
  cuuint64_t strides[2] = {row, row * (cuuint64_t)c.page_size};
  cuuint32_t box[3] = {(cuuint32_t)row, (cuuint32_t)(c.page_size < kChunk ? c.page_size : kChunk), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = c.head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WsLayout {
  size_t rec_off, ml_off, o_off, total;
};

WsLayout ws_layout(int64_t batch, int64_t hkv, int64_t g, int64_t d, int64_t ctas) {
  WsLayout L;
  const int64_t units = batch * hkv;
  const int64_t slots = units + ctas;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  L.rec_off = 0;
  L.ml_off = up((size_t)units * sizeof(int2));
  L.o_off = L.ml_off + up((size_t)slots * g * 2 * sizeof(float));
  L.total = L.o_off + up((size_t)slots * g * d * sizeof(float));
  return L;
}

int decode_ctas() { return 2 * device_sm_count(); }

template <int D>
kvq_status launch_decode(const kvq_cache& gc, const DecodeParams& dp, cudaStream_t s, int ctas) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return KVQ_ERR_CUDA;
  CUtensorMap tmk, tmv;
  if (!make_code_map(enc, &tmk, gc.k_codes, gc) || !make_code_map(enc, &tmv, gc.v_codes, gc))
    return KVQ_ERR_INVALID_ARGUMENT;
  const int smem = Geo<D>::kSmemBytes;
  if (cudaFuncSetAttribute(decode_fp4_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return KVQ_ERR_CUDA;
  decode_fp4_kernel<D><<<ctas, kThreads, smem, s>>>(tmk, tmv, dp);
  return launch_status();
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim) {
  if (batch < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0 ||
      head_dim < 16)
    return 0;
  const int ctas = decode_ctas();
  if (ctas <= 0) return 0;
  return ws_layout(batch, num_kv_heads, num_q_heads / num_kv_heads, head_dim, ctas).total;
}

extern "C" kvq_status kvq_decode_attn(const kvq_cache* global, const kvq_cache* swa, int32_t batch,
                                      int32_t num_q_heads, const int32_t* d_seq_lens, const void* q,
                                      float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                      int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 1) return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status st = check_cache(global, batch);
  if (st != KVQ_OK) return st;
  if (global->format != KVQ_FORMAT_FP4_E2M1_E4M3_G16) return KVQ_ERR_INVALID_ARGUMENT;
  const int hkv = global->num_kv_heads, D = global->head_dim;
  if (num_q_heads < hkv || num_q_heads % hkv != 0) return KVQ_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / hkv;
  if (!(softmax_scale > 0.0f) || !(softmax_scale < 3.0e38f)) return KVQ_ERR_INVALID_ARGUMENT;
  if (d_seq_lens == nullptr || q == nullptr || out == nullptr || workspace == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(q, 16) || !aligned_to(out, 16) || !aligned_to(workspace, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  if (swa != nullptr) {
    st = check_cache(swa, batch);
    if (st != KVQ_OK) return st;
    if (swa->format != KVQ_FORMAT_FP8_E4M3_HEAD || swa->num_kv_heads != hkv || swa->head_dim != D)
      return KVQ_ERR_INVALID_ARGUMENT;
  }
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (g > kNG) return KVQ_ERR_UNSUPPORTED;
  const int ctas = decode_ctas();
  if (ctas <= 0) return KVQ_ERR_CUDA;
  const WsLayout L = ws_layout(batch, hkv, g, D, ctas);
  if (workspace_bytes < L.total) return KVQ_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  DecodeParams dp;
  dp.lens = d_seq_lens;
  dp.page_table = global->page_table;
  dp.k_scales = static_cast<const uint8_t*>(global->k_scales);
  dp.v_scales = static_cast<const uint8_t*>(global->v_scales);
  dp.q = static_cast<const uint16_t*>(q);
  dp.part_o = reinterpret_cast<float*>(ws + L.o_off);
  dp.part_ml = reinterpret_cast<float*>(ws + L.ml_off);
  dp.unit_rec = reinterpret_cast<int2*>(ws + L.rec_off);
  dp.flag = d_err_flag;
  dp.num_pages = global->num_pages;
  dp.batch = batch;
  dp.hkv = hkv;
  dp.g = g;
  dp.hq = num_q_heads;
  dp.page = global->page_size;
  dp.max_pages = global->max_pages_per_seq;
  dp.window = swa ? swa->page_size : 0;
  dp.qk_log2 = softmax_scale * kLog2e;
  st = D == 128 ? launch_decode<128>(*global, dp, s, ctas) : launch_decode<64>(*global, dp, s, ctas);
  if (st != KVQ_OK) return st;

  MergeParams mp;
  mp.lens = d_seq_lens;
  mp.q = dp.q;
  mp.part_o = dp.part_o;
  mp.part_ml = dp.part_ml;
  mp.unit_rec = dp.unit_rec;
  mp.out = out;
  mp.flag = d_err_flag;
  mp.k8 = swa ? static_cast<const uint8_t*>(swa->k_codes) : nullptr;
  mp.v8 = swa ? static_cast<const uint8_t*>(swa->v_codes) : nullptr;
  mp.k8_scale = swa ? static_cast<const float*>(swa->k_scales) : nullptr;
  mp.v8_scale = swa ? static_cast<const float*>(swa->v_scales) : nullptr;
  mp.window = swa ? swa->page_size : 0;
  mp.hkv = hkv;
  mp.g = g;
  mp.hq = num_q_heads;
  mp.head_dim = D;
  mp.qk_log2 = dp.qk_log2;
  if (swa && swa->page_size > kMaxWindow) return KVQ_ERR_UNSUPPORTED;
  const int msmem = (kNG * D + kNG * (swa ? swa->page_size : 1) + 2 * kNG + kNG * D) * (int)sizeof(float);
  if (msmem > 48 * 1024 &&
      cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, msmem) != cudaSuccess)
    return KVQ_ERR_CUDA;
  merge_kernel<<<(unsigned)(batch * hkv), 128, msmem, s>>>(mp);
  return launch_status();
}
