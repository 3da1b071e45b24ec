// kvq_decode_kernel.cuh -- the split-K flash-decode attention kernel over
// the FP4 paged cache (mma.sync tensor-core products) and its launch
// templates.  kvq_decode.cu instantiates it with the library's fixed wait
// limit; kvq_decode_test_wait.cu instantiates it with the limit a test can
// shorten; kvq_merge.cu combines its per-range partials; kvq_decode_api.cu
// holds the C entry points.
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
// kv head h) pair is a unit; its FP4 positions are cut into chunks of 128
// tokens.  All units' chunks are laid end to end and the persistent grid
// (three CTAs per SM, two for small caches) splits that line into equal
// contiguous ranges, so ragged lengths balance to within one chunk.  A CTA
// writes one partial (m, l, o) per unit it touches; the merge kernel
// combines them.
//
// CTA = 4 consumer warps + 1 producer warp.  The pool stores each group of
// min(page, 128) tokens of one kv head as one contiguous block (K codes, K
// scales, V token-pair codes, V scales), so the producer's lane 0 fills a
// stage of the 3-stage ring with one or two cp.async.bulk copies, guarded by
// mbarriers (every wait bounded; a timeout sets a flag and the CTA exits in
// order).  Consumer warp w takes tokens [32w, 32w+32) of each chunk as two
// independent 16-token slices and runs, per slice:
//   S^T(16 tok x 8 q-rows) = K^(16 x d) Q^T    mma.m16n8k16, K^ dequantised in
//                                              registers (cvt e2m1x2->f16x2,
//                                              times the block scale)
//   online softmax in the log2 domain with lazy rescaling (the running max is
//   only raised when a score exceeds it by more than 8)
//   O^T(d x 8) += V^T(d x 16 tok) P^T           mma.m16n8k16, P in f16 moved
//                                              from the S^T fragment to the B
//                                              fragment with movmatrix.trans
// A stage's PV products go to fresh accumulators that are folded into O
// (rescaled only when the running max moved); the fused-append kernel
// accumulates them into O directly (see consume_stage).  Codes are expanded a 32-bit
// word (8 codes) at a time.  Each slice's K bytes are read from the stage
// right before its QK^T products and its V bytes right before its PV
// products; the stage goes back to the producer after the last slice's V
// loads.  (Reading the whole stage into registers first and releasing it
// early costs 40 live registers, which at three CTAs per SM pushed the
// kernel into spills.)  Tokens sit on the MMA's M side so a GQA group of
// up to 8 query heads fills N = 8 without padding rows.  The query is
// pre-scaled per head by a power of two so that its bf16 values are exact in
// f16; the factor is undone in fp32.
#pragma once
#include "kvq_append.cuh"
#include "kvq_common.cuh"
#include "kvq_decode.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kSlices = kChunk / (16 * kConsumerWarps);  // 16-token slices per warp per stage
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStages = 3;
constexpr int kMaxCopies = kChunk / 16;  // pool groups per stage at the smallest page size

// The kernel's work waits (a consumer waiting for a stage to land, the
// producer waiting for a free stage): the library's fixed ~2 s limit, or
// (TEST_WAIT, the instantiation used only while a test has shortened the
// limit) the limit carried in the parameters.  A separate instantiation keeps
// the production waits free of the runtime limit.
template <bool TEST_WAIT>
__device__ __forceinline__ bool work_wait(const DecodeParams& p, uint32_t bar, uint32_t parity) {
  if constexpr (TEST_WAIT)
    return mbar_wait_limit(bar, parity, p.wait_ns);
  else
    return mbar_wait(bar, parity);
}

template <int D>
struct Geo {
  // a stage holds kChunk tokens = kChunk / min(P, kChunk) consecutive pool groups
  static constexpr int kStageBytes = (kChunk * 9 * D / 8 + 1023) / 1024 * 1024;
  // flush buffer: O[warp][row][D], M[warp][row], L[warp][row]
  static constexpr int kFlushBytes = kConsumerWarps * kNG * (D + 2) * 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + kFlushBytes + 2 * kStages * 8 + kStages * 4 + 16 + 1024;
};

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
// Fused append (kvq_append_decode_attn): the newest token of unit (b, h),
// position T_b - 1, quantised and stored into the pool by the producer warp
// -- lanes 0 .. NQK-1 take the K items, the next NQV lanes the V item of its
// token pair -- exactly as kvq_append with one new token would; then every
// lane's stores are made visible to the bulk-copy (async) proxy before any
// later copy of the warp reads them.
template <int D>
__device__ void append_newest(const DecodeParams& p, int b, int h) {
  constexpr int NQK = D / 16 / kAppendBlocksK, NQV = D / 16 / kAppendBlocksV;
  const int lane = threadIdx.x & 31;
  if (lane < NQK + NQV) {
    const int64_t pos = (int64_t)__ldg(p.lens + b) - 1;
    const int64_t row = ((int64_t)b * p.hkv + h) * D;
    if (!KVQ_IN(b < p.batch && h < p.hkv, p.flag)) return;
    int ls = 0;
    if (lane < NQK) {
      const int j0 = lane * kAppendBlocksK;
      uint8_t* grp = fp4_group<D>(p.cache, b, pos, h, ls, p.flag);
      if (grp != nullptr) {
        if (p.nvfp4)
          append_k_item<D, true>(p.cache, grp, ls, h, j0, p.k_new + row + 16 * j0, p.flag);
        else
          append_k_item<D, false>(p.cache, grp, ls, h, j0, p.k_new + row + 16 * j0, p.flag);
      }
    } else {
      const int j0 = (lane - NQK) * kAppendBlocksV;
      uint8_t* grp = fp4_group<D>(p.cache, b, pos & ~(int64_t)1, h, ls, p.flag);
      if (grp != nullptr) {
        const bool even = (pos & 1) == 0;  // the new token is the pair's first (else its second)
        const uint16_t* src = p.v_new + row + 16 * j0;
        if (p.nvfp4)
          append_v_item<D, true>(p.cache, grp, ls, h, j0, even, !even, src, src, p.flag);
        else
          append_v_item<D, false>(p.cache, grp, ls, h, j0, even, !even, src, src, p.flag);
      }
    }
  }
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
  __syncwarp();
}

// Issue the bulk copies of one chunk into ring stage s (producer lane 0).
template <int D, int GT>
__device__ __forceinline__ void issue_chunk(const DecodeParams& p, Smem<D>& sm, const Walker& wk, uint32_t s) {
  using G = Geo<D>;
  using R = Grp<D, GT>;
  const int P = p.page;
  const int n4 = fp4_tokens(__ldg(p.lens + wk.b), p.window);
  const int tok0 = wk.c * kChunk;
  const int ntok = min(kChunk, n4 - tok0);
  // one copy per pool group: a 128-token group of a larger page, or whole small pages
  const int ncopies = GT < kChunk ? (ntok + GT - 1) / GT : 1;
  const int pg0 = tok0 / P;
  const int groups_per_page = P / GT;
  const int grp0 = GT < kChunk ? 0 : (tok0 % P) / GT;
  int64_t src[kMaxCopies];
  bool ok = true;
  for (int i = 0; i < ncopies; ++i) {
    const int pg = pg0 + i;
    int64_t ph = -1;
    if (pg < p.max_pages)
      ph = p.page_table ? (int64_t)__ldg(p.page_table + (int64_t)wk.b * p.max_pages + pg)
                        : (int64_t)wk.b * p.max_pages + pg;
    if (ph < 0 || ph >= p.num_pages) ok = false;
    src[i] = ((ph * p.hkv + wk.h) * groups_per_page + grp0) * (int64_t)R::kBytes;
    if (ok && !KVQ_IN(src[i] >= 0 && src[i] + R::kBytes <= p.pool_bytes && (i + 1) * R::kBytes <= G::kStageBytes,
                      p.flag))
      ok = false;
  }
  const uint32_t full = smem_addr(&sm.full[s]);
  uint8_t* st = sm.stages + s * G::kStageBytes;
  if (!ok) {
    set_flag(p.flag, KVQ_FLAG_PAGE_OOB);
    sm.ntok[s] = 0;
    mbar_arrive(full);
    return;
  }
  sm.ntok[s] = ntok;
  mbar_arrive_expect_tx(full, (uint32_t)(ncopies * R::kBytes));
  for (int i = 0; i < ncopies; ++i) bulk_g2s(smem_addr(st + i * R::kBytes), p.pool + src[i], R::kBytes, full);
}

// The producer warp.  Lane 0 waits for free ring stages and issues the bulk
// copies.  With a fused append (FUSED) the whole warp first stores the newest
// token of every unit whose last chunk lies in this CTA's range: the units
// ending in the first kStages chunks before those chunks are copied, the
// rest while those first copies are in flight, so the stores never hold up
// a refill of the ring.  The other lanes then leave and lane 0 goes on alone.
template <int D, int GT, bool FUSED, bool TEST_WAIT>
__device__ void producer(const DecodeParams& p, Smem<D>& sm, Walker wk, int64_t v1) {
  const int lane = threadIdx.x & 31;
  if (!FUSED && lane != 0) return;
  // launched as a programmatic dependent of the append kernel (the small-cache
  // path of kvq_append_decode_attn): the pool bytes are read only after that
  // grid has finished; otherwise this returns at once
  grid_dependency_wait();
  uint32_t it = 0;
  if (FUSED) {
    Walker aw = wk;
    for (int i = 0; i < kStages && aw.v < v1; ++i, advance(p, aw))
      if (aw.c == aw.nch - 1) append_newest<D>(p, aw.b, aw.h);
    for (; it < (uint32_t)kStages && wk.v < v1; advance(p, wk), ++it)
      if (lane == 0) issue_chunk<D, GT>(p, sm, wk, it);
    // the remaining unit ends of the range, one unit at a time
    while (aw.v < v1) {
      const int64_t last = aw.v + (aw.nch - 1 - aw.c);  // the unit's last chunk on the line
      if (last >= v1) break;
      append_newest<D>(p, aw.b, aw.h);
      aw.v = last;
      aw.c = aw.nch - 1;
      advance(p, aw);
    }
    if (lane != 0) return;
  }
  for (; wk.v < v1; advance(p, wk), ++it) {
    const uint32_t s = it % kStages;
    if (it >= (uint32_t)kStages) {
      if (!work_wait<TEST_WAIT>(p, smem_addr(&sm.empty[s]), ((it / kStages) + 1) & 1)) {
        set_flag(p.flag, KVQ_FLAG_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort) = 1;
        break;
      }
    }
    if (*reinterpret_cast<volatile int*>(sm.abort)) break;
    issue_chunk<D, GT>(p, sm, wk, s);
  }
  // Wait for every copy still in flight before the CTA can retire (the fixed
  // limit: copies always land, a shortened work-wait limit must not cut this).
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
  const int64_t qrow = (int64_t)b * p.hq + (int64_t)h * p.g + g;
  if (g < p.g && KVQ_IN(qrow < (int64_t)p.batch * p.hq, p.flag)) {
    const uint16_t* src = p.q + qrow * D + tig * kPer;
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
  // NVFP4: the keys' second-level scale multiplies every score of the head
  const float sk = p.k_gscale ? __ldg(p.k_gscale + h) : 1.0f;
  st.cs[0] = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - k0) << 23);
  st.cs[1] = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - k1) << 23);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mt][i] = 0.0f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.0f;
}

// One stage for one consumer warp: two 16-token slices, rows [32w, 32w+32).
// The stage holds pool groups of GT = min(page_size, 128) tokens back to back;
// a 16-token slice never straddles two groups.
// DIRECT: the stage's PV products accumulate straight into O (rescaled first
// when the running max moved) instead of into fresh accumulators folded into
// O afterwards.  The two forms compute the same sums in a different order;
// which one schedules better depends on the rest of the kernel: measured on
// long_context, DIRECT takes the fused-append kernel from 213.7 to 211.7 us
// and the plain one from 212.6 to 221.4 us, so the fused kernel uses it.
template <int D, int GT, bool PARTIAL, bool DIRECT>
__device__ __forceinline__ void consume_stage(ConsumerState<D>& st, uint32_t stage, int ntok,
                                              uint32_t empty_bar, int32_t* flag) {
  using G = Geo<D>;
  using R = Grp<D, GT>;
  constexpr int KW = D / 32;  // words of K codes per thread per row (channels [tig*D/4, +D/4))
  constexpr int VW = D / 32;  // words of V codes per thread per token pair (channels [g*D/8, +D/8))
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  // per-thread parts of the in-group offsets (pair rows i = lr/2 + tig have i % 8 == tig)
  const uint32_t k_lane = g * (D / 2) + tig * (D / 8);
  const uint32_t ks_lane = R::kKS + g * R::kNB + (D == 128 ? 2 * tig : tig);
  const uint32_t v_lane =
      R::kVC + tig * D + (D == 128 ? 16 * (g ^ (tig << 1)) : 8 * (g ^ (((tig >> 1) & 1) << 2)));
  const uint32_t vs_lane = R::kVS + tig * 2 * R::kNB + 2 * (D == 128 ? g : (g >> 1));

  // ---- S^T = K^ Q^T per slice (rows: tokens g, g+8; columns: q rows 2t, 2t+1);
  // each slice's K bytes are loaded right before its products
  float S[kSlices][4];
#pragma unroll
  for (int sl = 0; sl < kSlices; ++sl) {
    const int r0 = 16 * (kSlices * warp + sl);
    const uint32_t grp = stage + (uint32_t)((r0 / GT) * R::kBytes);
    const uint32_t lr = r0 % GT;
    uint32_t kp = grp + lr * (D / 2) + k_lane;
    uint32_t ksp = grp + lr * R::kNB + ks_lane;
    uint32_t kw[2][KW], ksb[2];
    // (bounds-checked build: a slice whose bytes would fall outside the stage
    // reads nothing and contributes zero codes)
    if (!KVQ_IN(kp + 8 * (D / 2) + D / 8 <= stage + G::kStageBytes && ksp + 8 * R::kNB + 2 <= stage + G::kStageBytes,
                flag)) {
      kp = ksp = stage;
    }
    if constexpr (D == 128) {
      const uint4 a = lds128(kp);
      const uint4 b = lds128(kp + 8 * (D / 2));
      kw[0][0] = a.x; kw[0][1] = a.y; kw[0][2] = a.z; kw[0][3] = a.w;
      kw[1][0] = b.x; kw[1][1] = b.y; kw[1][2] = b.z; kw[1][3] = b.w;
      ksb[0] = lds16(ksp);
      ksb[1] = lds16(ksp + 8 * R::kNB);
    } else {
      const uint2 a = lds64(kp);
      const uint2 b = lds64(kp + 8 * (D / 2));
      kw[0][0] = a.x; kw[0][1] = a.y;
      kw[1][0] = b.x; kw[1][1] = b.y;
      ksb[0] = lds8(ksp);
      ksb[1] = lds8(ksp + 8 * R::kNB);
    }
    uint32_t sc[2][2];  // [row g / g+8][first / second block of the thread's channels]
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if constexpr (D == 128) {
        const uint32_t u = f16x2_from_e4m3x2(ksb[r]);
        sc[r][0] = prmt(u, 0u, 0x1010u);
        sc[r][1] = prmt(u, 0u, 0x3232u);
      } else {
        sc[r][0] = sc[r][1] = f16x2_from_e4m3x2(ksb[r] * 0x0101u);
      }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < KW; ++q) {  // word q holds k-steps 2q (bytes 0,1) and 2q+1 (bytes 2,3)
      uint32_t ca[4], cb[4];
      f16x2x4_from_e2m1x8(kw[0][q], ca);
      f16x2x4_from_e2m1x8(kw[1][q], cb);
      const int half = (D == 128 && q >= KW / 2) ? 1 : 0;
      const uint32_t sA = sc[0][half], sB = sc[1][half];
      mma_f16_16816(acc, hmul2_u32(ca[0], sA), hmul2_u32(cb[0], sB), hmul2_u32(ca[1], sA),
                    hmul2_u32(cb[1], sB), st.qf[4 * q], st.qf[4 * q + 1]);
      mma_f16_16816(acc, hmul2_u32(ca[2], sA), hmul2_u32(cb[2], sB), hmul2_u32(ca[3], sA),
                    hmul2_u32(cb[3], sB), st.qf[4 * q + 2], st.qf[4 * q + 3]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) S[sl][i] = acc[i];
  }
  // PARTIAL: the stage holds fewer than kChunk tokens (only a unit's last
  // chunk); full stages get code without any of the masking below
  constexpr bool partial = PARTIAL;
  if (partial) {
#pragma unroll
    for (int sl = 0; sl < kSlices; ++sl) {
      const int t0 = 16 * (kSlices * warp + sl) + g;
      if (t0 >= ntok) S[sl][0] = S[sl][1] = -INFINITY;
      if (t0 + 8 >= ntok) S[sl][2] = S[sl][3] = -INFINITY;
    }
  }

  // ---- online softmax in the log2 domain (cs > 0, so the max commutes with the scale)
  float m0 = fmaxf(S[0][0], S[0][2]), m1 = fmaxf(S[0][1], S[0][3]);
#pragma unroll
  for (int sl = 1; sl < kSlices; ++sl) {
    m0 = fmaxf(m0, fmaxf(S[sl][0], S[sl][2]));
    m1 = fmaxf(m1, fmaxf(S[sl][1], S[sl][3]));
  }
  m0 *= st.cs[0];
  m1 *= st.cs[1];
  // O is rescaled (by al) when this stage's products are added to it, below
  float al0 = 1.0f, al1 = 1.0f;
  const bool rescale = __any_sync(0xFFFFFFFFu, m0 > st.m[0] + kLazySlack || m1 > st.m[1] + kLazySlack);
  if (rescale) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, o));
    }
    const float n0 = fmaxf(st.m[0], m0), n1 = fmaxf(st.m[1], m1);
    al0 = (st.m[0] == -INFINITY) ? 0.0f : fast_exp2(st.m[0] - n0);
    al1 = (st.m[1] == -INFINITY) ? 0.0f : fast_exp2(st.m[1] - n1);
    st.l[0] *= al0;
    st.l[1] *= al1;
    st.m[0] = n0;
    st.m[1] = n1;
  }
  const float nref0 = st.m[0] == -INFINITY ? 0.0f : -st.m[0];
  const float nref1 = st.m[1] == -INFINITY ? 0.0f : -st.m[1];

  float acc[D / 16][4];  // this stage's PV products (fresh accumulators; unused when DIRECT)
  if constexpr (DIRECT) {
    if (rescale) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        st.o[mt][0] *= al0;
        st.o[mt][1] *= al1;
        st.o[mt][2] *= al0;
        st.o[mt][3] *= al1;
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
  }
#pragma unroll
  for (int sl = 0; sl < kSlices; ++sl) {
    const float p0 = fast_exp2(fmaf(S[sl][0], st.cs[0], nref0));
    const float p1 = fast_exp2(fmaf(S[sl][1], st.cs[1], nref1));
    const float p2 = fast_exp2(fmaf(S[sl][2], st.cs[0], nref0));
    const float p3 = fast_exp2(fmaf(S[sl][3], st.cs[1], nref1));
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    // P^T B fragment: k-slots (2t, 2t+1) <- tokens 2t, 2t+1; (2t+8, 2t+9) <- 2t+8, 2t+9
    const uint32_t pbA = movmatrix_trans(pack_f16x2(p0, p1));
    const uint32_t pbB = movmatrix_trans(pack_f16x2(p2, p3));

    // ---- O^T += V^T P^T: this slice's V bytes, then (after the last slice)
    // the stage goes back to the producer
    const int r0v = 16 * (kSlices * warp + sl);
    const uint32_t grpv = stage + (uint32_t)((r0v / GT) * R::kBytes);
    const uint32_t lrv = r0v % GT;
    uint32_t vp = grpv + (lrv / 2) * D + v_lane;
    uint32_t vsp = grpv + (lrv / 2) * 2 * R::kNB + vs_lane;
    if (!KVQ_IN(vp + 4 * D + D / 8 <= stage + G::kStageBytes && vsp + 8 * R::kNB + 2 <= stage + G::kStageBytes,
                flag)) {
      vp = vsp = stage;
    }
    uint32_t vwl[2][VW];
    if constexpr (D == 128) {
      const uint4 x = lds128(vp);
      const uint4 y = lds128(vp + 4 * D);  // pair row i + 4: same permutation
      vwl[0][0] = x.x; vwl[0][1] = x.y; vwl[0][2] = x.z; vwl[0][3] = x.w;
      vwl[1][0] = y.x; vwl[1][1] = y.y; vwl[1][2] = y.z; vwl[1][3] = y.w;
    } else {
      const uint2 x = lds64(vp);
      const uint2 y = lds64(vp + 4 * D);  // (i + 4) >> 1 keeps bit 0
      vwl[0][0] = x.x; vwl[0][1] = x.y;
      vwl[1][0] = y.x; vwl[1][1] = y.y;
    }
    uint32_t vsA = lds16(vsp), vsB = lds16(vsp + 4 * 2 * R::kNB);
    if (sl == kSlices - 1) mbar_arrive(empty_bar);
    if (partial) {  // masked tokens get a zero V scale so stale bytes cannot inject NaN
      const int t0 = 16 * (kSlices * warp + sl) + 2 * tig;
      if (t0 >= ntok) vsA &= 0xFF00u;
      if (t0 + 1 >= ntok) vsA &= 0x00FFu;
      if (t0 + 8 >= ntok) vsB &= 0xFF00u;
      if (t0 + 9 >= ntok) vsB &= 0x00FFu;
    }
    const uint32_t svA = f16x2_from_e4m3x2(vsA);
    const uint32_t svB = f16x2_from_e4m3x2(vsB);
    // byte c of a pair row = channel c of tokens (2t, 2t+1) -> f16x2 (low, high)
    uint32_t VA[4 * VW], VB[4 * VW];
#pragma unroll
    for (int w = 0; w < VW; ++w) {
      uint32_t ta[4], tb[4];
      f16x2x4_from_e2m1x8(vwl[0][w], ta);
      f16x2x4_from_e2m1x8(vwl[1][w], tb);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        VA[4 * w + k] = ta[k];
        VB[4 * w + k] = tb[k];
      }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      // row g <-> channel (D/8) g + mt, row g+8 <-> (D/8) g + D/16 + mt
      const uint32_t a0 = hmul2_u32(VA[mt], svA), a1 = hmul2_u32(VA[D / 16 + mt], svA);
      const uint32_t a2 = hmul2_u32(VB[mt], svB), a3 = hmul2_u32(VB[D / 16 + mt], svB);
      if constexpr (DIRECT)
        mma_f16_16816(st.o[mt], a0, a1, a2, a3, pbA, pbB);
      else
        mma_f16_16816(acc[mt], a0, a1, a2, a3, pbA, pbB);
    }
  }
  if constexpr (DIRECT) return;
  if (rescale) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.o[mt][0] = fmaf(st.o[mt][0], al0, acc[mt][0]);
      st.o[mt][1] = fmaf(st.o[mt][1], al1, acc[mt][1]);
      st.o[mt][2] = fmaf(st.o[mt][2], al0, acc[mt][2]);
      st.o[mt][3] = fmaf(st.o[mt][3], al1, acc[mt][3]);
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[mt][i] += acc[mt][i];
  }
}

// Combine the four warps' states for one unit and write the CTA's partial.
template <int D>
__device__ void flush_unit(const DecodeParams& p, ConsumerState<D>& st, Smem<D>& sm, int64_t slot, float vscale) {
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
    if (!KVQ_IN(slot >= 0 && slot < p.n_slots, p.flag)) continue;
    p.part_o[(slot * p.g + r) * D + ch] = o * vscale;  // NVFP4: the values' second-level scale
    if (ch == 0) {
      p.part_ml[(slot * p.g + r) * 2 + 0] = mx;
      p.part_ml[(slot * p.g + r) * 2 + 1] = l;
    }
  }
}

template <int D, int GT, bool FUSED, bool TEST_WAIT>
__global__ void __launch_bounds__(kThreads, 3)
    decode_fp4_kernel(const DecodeParams p) {
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
  // The merge grid is launched as a programmatic dependent and waits for
  // this grid's results before reading them.  With an FP8 window it has
  // work of its own (the window's scores and PV products) that overlaps
  // this grid's tail only if it is released now: swa_append 222.9 -> 215.3
  // us.  Without a window it has nothing to do before the wait, and
  // releasing it at each CTA's exit instead is faster: long_context's fused
  // step 211.3 -> 209.6 us.
  if (p.window > 0) grid_launch_dependents();
  plan(p, blockIdx.x, gridDim.x, total, v0, v1, wk);
  if (v0 >= v1) return;

  if (warp == kConsumerWarps) {
    producer<D, GT, FUSED, TEST_WAIT>(p, sm, wk, v1);
    return;
  }

  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const uint32_t stages_base = smem_addr(sm.stages);
  ConsumerState<D> st;
  bool have = false, dead = false;
  int64_t slot = 0;
  float vscale = 1.0f;
  uint32_t it = 0;
  for (; wk.v < v1; advance(p, wk), ++it) {
    if (!have || wk.c == 0) {
      if (have) flush_unit<D>(p, st, sm, slot, vscale);
      const int64_t u = (int64_t)wk.b * p.hkv + wk.h;
      vscale = p.v_gscale ? __ldg(p.v_gscale + wk.h) : 1.0f;
      slot = u + blockIdx.x;
      begin_unit<D>(p, st, wk.b, wk.h);
      have = true;
      if (wk.c == 0 && threadIdx.x == 0) {
        const int64_t last_cta = (wk.v + wk.nch - 1) / per;
        if (KVQ_IN(u < (int64_t)p.batch * p.hkv && last_cta < gridDim.x, p.flag))
          p.unit_rec[u] = make_int2((int)slot, (int)(last_cta - blockIdx.x + 1));
      }
    }
    if (dead) continue;
    const uint32_t s = it % kStages;
    bool ok = !*reinterpret_cast<volatile int*>(sm.abort) &&
              work_wait<TEST_WAIT>(p, smem_addr(&sm.full[s]), (it / kStages) & 1);
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
    if (ntok > 16 * kSlices * warp) {
      if (ntok < kChunk)
        consume_stage<D, GT, true, FUSED>(st, stages_base + s * G::kStageBytes, ntok, smem_addr(&sm.empty[s]),
                                          p.flag);
      else
        consume_stage<D, GT, false, FUSED>(st, stages_base + s * G::kStageBytes, ntok, smem_addr(&sm.empty[s]),
                                           p.flag);
    } else {
      mbar_arrive(smem_addr(&sm.empty[s]));
    }
  }
  if (have) flush_unit<D>(p, st, sm, slot, vscale);
}

template <int D, int GT, bool FUSED, bool TEST_WAIT>
kvq_status launch_decode_f(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append) {
  const int smem = Geo<D>::kSmemBytes;
  static DeviceOnce attr_set;  // the shared-memory opt-in, once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(decode_fp4_kernel<D, GT, FUSED, TEST_WAIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  if (!after_append) {
    decode_fp4_kernel<D, GT, FUSED, TEST_WAIT><<<ctas, kThreads, smem, s>>>(dp);
    return launch_status();
  }
  // a programmatic dependent of the append kernel just enqueued
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fp4_kernel<D, GT, FUSED, TEST_WAIT>, dp) == cudaSuccess ? KVQ_OK
                                                                                           : KVQ_ERR_CUDA;
}

template <int D, int GT, bool TEST_WAIT>
kvq_status launch_decode_g(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append) {
  return dp.k_new != nullptr ? launch_decode_f<D, GT, true, TEST_WAIT>(dp, s, ctas, after_append)
                             : launch_decode_f<D, GT, false, TEST_WAIT>(dp, s, ctas, after_append);
}

template <int D, bool TEST_WAIT>
kvq_status launch_decode(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append) {
  switch (dp.page < kChunk ? dp.page : kChunk) {
    case 16: return launch_decode_g<D, 16, TEST_WAIT>(dp, s, ctas, after_append);
    case 32: return launch_decode_g<D, 32, TEST_WAIT>(dp, s, ctas, after_append);
    case 64: return launch_decode_g<D, 64, TEST_WAIT>(dp, s, ctas, after_append);
    default: return launch_decode_g<D, kChunk, TEST_WAIT>(dp, s, ctas, after_append);
  }
}

}  // namespace
}  // namespace kvq
