// kvq_decode_tc.cu -- split-K flash-decode attention over the FP4 paged cache
// for head_dim 128, with both products on the 5th-generation tensor cores
// (tcgen05, operands and accumulators in tensor memory).
//
// Method: "Quantising the KV cache", section "Code" -- the quantised K and V
// feed an unchanged attention, out = softmax(scale * q.K^T) V^ -- and
// "KV Cache Quantisation", section "Common questions": the kernel does the
// scale handling itself; codes and scales are read once from HBM and expanded
// in registers, and the expanded values go straight to tensor memory, never
// back to shared memory.
//
// Work decomposition: the same stream-K line of 128-token chunks as the
// mma.sync kernel (kvq_decode.cu), cut into 3 x (number of SMs) equal ranges;
// the same per-range partials and the same merge kernels.  One CTA per SM runs
// three independent pipelines ("warpgroups"), each owning one range, 160
// columns of tensor memory and its own 3-stage ring of bulk copies:
//   producer warp (lane 0)  cp.async.bulk of the pool groups of each chunk
//   4 consumer warps        per 128-token stage:
//     K^ (token split)      warp w expands tokens [32w, 32w+32) (E2M1 code
//                           times E4M3 scale, f16) and stores them with
//                           tcgen05.st.16x256b into TMEM lanes = tokens;
//     S = K^ Q^T            one thread issues 8 x tcgen05.mma M=128 N=16 K=16
//                           (A = K^ from TMEM, B = the query tile in shared
//                           memory, 8 query rows padded to 16), D = S in TMEM;
//     V^T (channel split)   warp w expands channels [32w, 32w+32) of all 128
//                           tokens into TMEM lanes = channels (overlapping the
//                           S products);
//     softmax               S read back with tcgen05.ld.16x256b (the mma
//                           fragment layout), online softmax in the log2
//                           domain with a lazy running max shared by the
//                           warpgroup (raised only when a score passes it by
//                           more than 8; one barrier reduction per stage
//                           decides), P = 2^(s - m) as f16 into a shared
//                           memory tile (the B operand, K-major);
//     O^T += V^T P^T        8 x tcgen05.mma M=128 N=16 K=16, O in TMEM
//                           (rescaled in TMEM on the rare raise of the max).
// At the end of a unit the warpgroup reads O from TMEM and writes its partial
// (m, l, o) like the mma.sync kernel.  Every wait is bounded; on a timeout the
// warpgroup stops (all its threads together), waits for its own MMAs, and the
// CTA frees its TMEM before it exits.
#include "kvq_common.cuh"
#include "kvq_decode.cuh"
#include "kvq_host.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kTD = 128;                            // head_dim of this kernel
constexpr int kTWG = 3;                             // pipelines per CTA
constexpr int kTStages = 3;                         // ring stages per pipeline
constexpr int kTN = 16;                             // MMA N (query rows padded to 16)
constexpr int kTThreads = 32 * (4 * kTWG + kTWG);   // 12 consumer warps, then 3 producer warps
constexpr int kTStageBytes = kChunk * 9 * kTD / 8;  // one 128-token stage of one kv head
constexpr int kTOpBytes = kTN * kTD * 2;            // the query or P tile: 16 rows x 128 f16
constexpr int kTMaxCopies = kChunk / 16;
// TMEM columns of one pipeline: K^ [tokens][channels] f16 pairs, V^T
// [channels][tokens] f16 pairs, S [tokens][16] fp32, O [channels][16] fp32
constexpr uint32_t kColK = 0, kColV = 64, kColS = 128, kColO = 144, kColsPerWG = 160;
constexpr uint32_t kTTmemCols = 512;

// Shared memory of one pipeline (offsets from its base).
struct TcWG {
  static constexpr int kStage = 0;                              // [kTStages][kTStageBytes]
  static constexpr int kQ = kStage + kTStages * kTStageBytes;   // query tile (B of S = K^ Q^T)
  static constexpr int kP = kQ + kTOpBytes;                     // P tile (B of O^T += V^T P^T)
  static constexpr int kRedMax = kP + kTOpBytes;                // float [4 warps][8 rows]
  static constexpr int kRedL = kRedMax + 128;                   // float [4 warps][8 rows]
  static constexpr int kKexp = kRedL + 128;                     // int [8]: query prescale exponents
  static constexpr int kBar = kKexp + 32;                       // full[3], empty[3], s_full, pv_done
  static constexpr int kNtok = kBar + 8 * (2 * kTStages + 2);   // int [kTStages]
  static constexpr int kAbort = kNtok + 4 * kTStages;           // int: the consumers gave up
  static constexpr int kBytes = (kAbort + 4 + 127) / 128 * 128;
  static_assert(kQ % 128 == 0 && kP % 128 == 0 && kBar % 8 == 0, "pipeline shared-memory alignment");
};
constexpr int kTSmemBytes = kTWG * TcWG::kBytes + 128 + 1024;  // + TMEM slot, + alignment slack
static_assert(kTSmemBytes <= 227 * 1024, "shared memory per CTA");

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ void wg_bar(uint32_t id) { named_barrier_sync(id, 128); }

// Barrier of the warpgroup's 128 threads that also ORs a predicate over them.
__device__ __forceinline__ bool wg_bar_or(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id)
      : "memory");
  return r != 0;
}

// 8 repetitions of the 16-lane x 256-bit TMEM access (the mma fragment
// layout): repetition r covers columns [8r, 8r+8); thread (g, t) holds
// v[4r..4r+3] = (lane g: column 8r+2t, 8r+2t+1; lane g+8: the same columns).
__device__ __forceinline__ void tmem_st_16x256b_x8(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// One repetition of the same shape, loaded (fp32 accumulators).
__device__ __forceinline__ void tmem_ld_16x256b_x1(uint32_t taddr, float (&v)[4]) {
  uint32_t r0, r1, r2, r3;
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(taddr)
               : "memory");
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2);
  v[3] = __uint_as_float(r3);
}
// 8 consecutive columns of this warp's 32 lanes (thread = lane), and the store.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_only() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// E2M1 byte k of a word -> f16x2 (low nibble -> low half).
template <int K>
__device__ __forceinline__ uint32_t f16x2_from_e2m1_byte(uint32_t w) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b" "%2" ";\n}\n"
      : "=r"(r)
      : "r"(w), "n"(K));
  return r;
}

// Channel of TMEM lane L (0..127) in the V^T / O operand: warp w's lanes
// 32w + 16s + 8a + g hold channel 32w + 4g + 2s + a, so that thread (g, t)
// of warp w stores the four channels 32w + 4g .. +3 (one block).
__device__ __forceinline__ int vlane_channel(int L) {
  return (L & ~31) + 4 * (L & 7) + 2 * ((L >> 4) & 1) + ((L >> 3) & 1);
}

// ---------------------------------------------------------------- producer
template <int GT>
__device__ void tc_producer(const DecodeParams& p, uint8_t* wb, uint32_t wsb, Walker wk, int64_t v1) {
  using R = Grp<kTD, GT>;
  const int P = p.page;
  int* ntok_s = reinterpret_cast<int*>(wb + TcWG::kNtok);
  volatile int* cons_abort = reinterpret_cast<volatile int*>(wb + TcWG::kAbort);
  const uint32_t full0 = wsb + TcWG::kBar, empty0 = full0 + 8 * kTStages;
  uint32_t it = 0;
  for (; wk.v < v1; advance(p, wk), ++it) {
    const uint32_t s = it % kTStages;
    if (it >= (uint32_t)kTStages) {
      if (!mbar_wait(empty0 + 8 * s, ((it / kTStages) + 1) & 1)) {
        set_flag(p.flag, KVQ_FLAG_TIMEOUT);
        break;
      }
    }
    if (*cons_abort) break;
    const int n4 = fp4_tokens(__ldg(p.lens + wk.b), p.window);
    const int tok0 = wk.c * kChunk;
    const int ntok = min(kChunk, n4 - tok0);
    const int ncopies = GT < kChunk ? (ntok + GT - 1) / GT : 1;
    const int pg0 = tok0 / P;
    const int groups_per_page = P / GT;
    const int grp0 = GT < kChunk ? 0 : (tok0 % P) / GT;
    int64_t src[kTMaxCopies];
    bool ok = true;
    for (int i = 0; i < ncopies; ++i) {
      const int pg = pg0 + i;
      int64_t ph = -1;
      if (pg < p.max_pages)
        ph = p.page_table ? (int64_t)__ldg(p.page_table + (int64_t)wk.b * p.max_pages + pg)
                          : (int64_t)wk.b * p.max_pages + pg;
      if (ph < 0 || ph >= p.num_pages) ok = false;
      src[i] = ((ph * p.hkv + wk.h) * groups_per_page + grp0) * (int64_t)R::kBytes;
    }
    const uint32_t full = full0 + 8 * s;
    const uint32_t st = wsb + TcWG::kStage + s * kTStageBytes;
    if (!ok) {
      set_flag(p.flag, KVQ_FLAG_PAGE_OOB);
      ntok_s[s] = 0;
      mbar_arrive(full);
      continue;
    }
    ntok_s[s] = ntok;
    mbar_arrive_expect_tx(full, (uint32_t)(ncopies * R::kBytes));
    for (int i = 0; i < ncopies; ++i) bulk_g2s(st + i * R::kBytes, p.pool + src[i], R::kBytes, full);
  }
  // every copy still in flight lands before the CTA can retire
  const uint32_t first = it > (uint32_t)kTStages ? it - kTStages : 0;
  for (uint32_t j = first; j < it; ++j) {
    if (!mbar_wait(full0 + 8 * (j % kTStages), (j / kTStages) & 1)) {
      set_flag(p.flag, KVQ_FLAG_TIMEOUT);
      break;
    }
  }
}

// ---------------------------------------------------------------- consumers
struct TcState {
  float cs[2];    // score scale (softmax scale * log2 e * query prescale) of rows 2t, 2t+1
  float m[2];     // running max of rows 2t, 2t+1 (the same in every thread of the warpgroup)
  float mall[8];  // the running max of every row (for the rescale of O)
  float l[2];     // this thread's share of the row sums of rows 2t, 2t+1
};

// The query tile of unit (b, h) into the B operand of S = K^ Q^T: row n (query
// head h*G + n; rows >= G and 8..15 zero) and 128 channels in the tensor
// core's K-major core layout, the K index permuted to match the K^ columns
// (column 16q + 8e + 2t + k of K^ holds channel pair 16t + 4q + 2e + k).  Each
// row is prescaled by a power of two so that its bf16 values are exact in f16;
// the exponent goes to kexp[n] and returns in the score scale.  Thread i (of
// 128) writes row i / 16, K indices [8 (i % 16), +8).
__device__ __forceinline__ void tc_load_query(const DecodeParams& p, uint32_t qbuf, int* kexp, int b, int h, int i) {
  const int n = i >> 4, kc = i & 15;
  const int ch0 = 2 * (32 * (kc & 1) + 4 * (kc >> 2) + 2 * ((kc >> 1) & 1));
  uint2 a = make_uint2(0u, 0u), c = make_uint2(0u, 0u);
  if (n < p.g) {
    const uint16_t* src = p.q + ((int64_t)b * p.hq + (int64_t)h * p.g + n) * kTD;
    a = __ldg(reinterpret_cast<const uint2*>(src + ch0));
    c = __ldg(reinterpret_cast<const uint2*>(src + ch0 + 32));
  }
  const uint32_t w4[4] = {a.x, a.y, c.x, c.y};
  uint32_t amax_bits = 0u;  // |x| of the row's largest element (bf16 bits, upper half)
#pragma unroll
  for (int k = 0; k < 4; ++k) amax_bits = max(amax_bits, max((w4[k] << 16) & 0x7FFF0000u, w4[k] & 0x7FFF0000u));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
  const float amax = __uint_as_float(amax_bits);
  int k = 0;  // max |q| * 2^k in [2^14, 2^15): bf16 values stay exact in f16
  if (amax > 0.0f && amax <= 3.4e38f) {
    const int e = (int)((amax_bits >> 23) & 0xFF) - 127;
    k = min(100, max(-113, 14 - e));
  }
  const float up = __uint_as_float((uint32_t)(k + 127) << 23);
  uint32_t f[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = pack_f16x2(bf16_lo(w4[j]) * up, bf16_hi(w4[j]) * up);
  sts128(qbuf + core_offset((uint32_t)n, (uint32_t)(8 * kc), kTN), make_uint4(f[0], f[1], f[2], f[3]));
  fence_async_smem();
  if (kc == 0) kexp[n] = k;
}

template <int GT>
__device__ void tc_consumer(const DecodeParams& p, uint8_t* wb, uint32_t wsb, uint32_t tmem_wg, int wg, Walker wk,
                            int64_t v1, int64_t total, int vidx, int vcount) {
  using R = Grp<kTD, GT>;
  constexpr int kNB = kTD / 16;
  const int i = threadIdx.x & 127;  // thread of the warpgroup
  const int w = i >> 5, lane = i & 31, g = lane >> 2, t = lane & 3;
  const uint32_t idA = 1 + 2 * wg, idB = 2 + 2 * wg;  // named barriers of this warpgroup
  const uint32_t full0 = wsb + TcWG::kBar, empty0 = full0 + 8 * kTStages;
  const uint32_t s_full = empty0 + 8 * kTStages, pv_done = s_full + 8;
  const uint32_t qbuf = wsb + TcWG::kQ, pbuf = wsb + TcWG::kP;
  float* red_max = reinterpret_cast<float*>(wb + TcWG::kRedMax);
  float* red_l = reinterpret_cast<float*>(wb + TcWG::kRedL);
  int* kexp = reinterpret_cast<int*>(wb + TcWG::kKexp);
  const int* ntok_s = reinterpret_cast<const int*>(wb + TcWG::kNtok);
  volatile int* abort = reinterpret_cast<volatile int*>(wb + TcWG::kAbort);
  const uint32_t tw = tmem_wg + ((uint32_t)(32 * w) << 16);  // this warp's TMEM lanes
  constexpr uint32_t kIdesc = idesc_f16_f32(128, kTN);
  const uint64_t qdesc = smem_desc(qbuf, (kTN / 8) * 128, 128);
  const uint64_t pdesc = smem_desc(pbuf, (kTN / 8) * 128, 128);
  const int64_t per = (total + vcount - 1) / vcount;

  TcState st = {};
  bool have = false, new_unit = false, first_pv = true;
  int64_t slot = 0;
  float vscale = 1.0f;
  uint32_t it = 0, sidx = 0, sphase = 0;  // stages consumed; ring slot and its phase parity
  uint32_t n_pv = 0, n_qk = 0;            // MMA batches committed (their barriers' phase counts)
  bool failed = false;

  // ---- the partial of the unit just finished: O from TMEM, m and l
  auto flush = [&]() {
    if (n_pv > 0 && !mbar_wait(pv_done, (n_pv - 1) & 1)) failed = true;
    tc_fence_after();
    float o[8];
    tmem_ld_32x32b_x8(tw + kColO, o);
    tmem_wait_ld_only();
    const int ch = vlane_channel(32 * w + lane);
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
    }
    if (g == 0) {
      red_l[w * 8 + 2 * t] = l0;
      red_l[w * 8 + 2 * t + 1] = l1;
    }
#pragma unroll
    for (int r = 0; r < kNG; ++r)
      if (r < p.g) p.part_o[(slot * p.g + r) * kTD + ch] = o[r] * vscale;
    wg_bar(idA);
    if (w == 0 && g == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 2 * t + e;
        if (r < p.g) {
          const float l = red_l[r] + red_l[8 + r] + red_l[16 + r] + red_l[24 + r];
          p.part_ml[(slot * p.g + r) * 2 + 0] = st.m[e];
          p.part_ml[(slot * p.g + r) * 2 + 1] = l;
        }
      }
    }
  };

  for (; wk.v < v1; advance(p, wk)) {
    if (!have || wk.c == 0) {
      if (have) flush();
      const int64_t u = (int64_t)wk.b * p.hkv + wk.h;
      vscale = p.v_gscale ? __ldg(p.v_gscale + wk.h) : 1.0f;
      slot = u + vidx;
      tc_load_query(p, qbuf, kexp, wk.b, wk.h, i);
      st.m[0] = st.m[1] = -INFINITY;
#pragma unroll
      for (int r = 0; r < 8; ++r) st.mall[r] = -INFINITY;
      st.l[0] = st.l[1] = 0.0f;
      have = true;
      new_unit = true;
      first_pv = true;
      if (wk.c == 0 && i == 0) {
        const int64_t last = (wk.v + wk.nch - 1) / per;
        p.unit_rec[u] = make_int2((int)slot, (int)(last - vidx + 1));
      }
    }
    // ---- the stage has landed
    if (!mbar_wait(full0 + 8 * sidx, sphase)) failed = true;
    const int ntok = ntok_s[sidx];
    const uint32_t stage = wsb + TcWG::kStage + sidx * kTStageBytes;

    // ---- K^: this warp's tokens [32w, 32w+32) as two 16-lane groups
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) {
      const int r0 = 32 * w + 16 * sl;
      const uint32_t grp = stage + (uint32_t)((r0 / GT) * R::kBytes);
      const uint32_t lr = (uint32_t)(r0 % GT) + g;
      const uint32_t kp = grp + lr * (kTD / 2) + t * (kTD / 8);
      const uint32_t ksp = grp + R::kKS + lr * kNB + 2 * t;
      const uint4 ka = lds128(kp), kb = lds128(kp + 8 * (kTD / 2));
      const uint32_t ua = f16x2_from_e4m3x2(lds16(ksp)), ub = f16x2_from_e4m3x2(lds16(ksp + 8 * kNB));
      const uint32_t sa[2] = {prmt(ua, 0u, 0x1010u), prmt(ua, 0u, 0x3232u)};
      const uint32_t sb[2] = {prmt(ub, 0u, 0x1010u), prmt(ub, 0u, 0x3232u)};
      const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wbw[4] = {kb.x, kb.y, kb.z, kb.w};
      uint32_t v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // word q: channels 32t + 8q .. +7 (block 2t + q / 2)
        uint32_t ca[4], cb[4];
        f16x2x4_from_e2m1x8(wa[q], ca);
        f16x2x4_from_e2m1x8(wbw[q], cb);
        const int hs = q >> 1;
#pragma unroll
        for (int e = 0; e < 2; ++e) {  // repetition 2q + e: columns 16q + 8e + 2t, +1
          v[4 * (2 * q + e) + 0] = hmul2_u32(ca[2 * e], sa[hs]);
          v[4 * (2 * q + e) + 1] = hmul2_u32(ca[2 * e + 1], sa[hs]);
          v[4 * (2 * q + e) + 2] = hmul2_u32(cb[2 * e], sb[hs]);
          v[4 * (2 * q + e) + 3] = hmul2_u32(cb[2 * e + 1], sb[hs]);
        }
      }
      tmem_st_16x256b_x8(tw + ((uint32_t)(16 * sl) << 16) + kColK, v);
    }
    tmem_wait_st();
    tc_fence_before();
    if (wg_bar_or(idA, failed)) {  // a wait gave up somewhere in the warpgroup: stop together
      failed = true;
      break;
    }
    if (new_unit) {  // the query prescale exponents of the new unit are published
      const float sk = p.k_gscale ? __ldg(p.k_gscale + wk.h) : 1.0f;
      st.cs[0] = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - kexp[2 * t]) << 23);
      st.cs[1] = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - kexp[2 * t + 1]) << 23);
      new_unit = false;
    }
    if (i == 0) {  // S = K^ Q^T
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTD / 16; ++ks)
        tc_mma_f16_ta(tmem_wg + kColS, tmem_wg + kColK + 8 * ks, qdesc + (uint64_t)(ks * 2 * (kTN / 8) * 8), kIdesc,
                      ks > 0);
      tc_commit(s_full);
    }
    ++n_qk;

    // ---- V^T: channels 32w + 4g .. +3 (block 2w + g / 4) of token pairs
    // 8r + 4e + t (r = 0..7, e = 0, 1): column 8r + 2t + e
    uint32_t vw[16], vs[16];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pr = 8 * r + 4 * e + t;  // token pair of the stage
        const uint32_t grp = stage + (uint32_t)(((2 * pr) / GT) * R::kBytes);
        const uint32_t lp = (uint32_t)(pr % (GT / 2));
        const uint32_t u = (uint32_t)(2 * w + (g >> 2));  // 16-byte chunk of the channels
        vw[2 * r + e] = lds32(grp + R::kVC + lp * kTD + ((u ^ ((lp & 3u) << 1)) << 4) + 4 * (g & 3));
        vs[2 * r + e] = lds16(grp + R::kVS + lp * 2 * kNB + 2 * u);
      }
    mbar_arrive(empty0 + 8 * sidx);  // the stage's bytes are all in registers
    if (ntok < kChunk) {             // masked tokens get a zero V scale (stale bytes cannot inject NaN)
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t0 = 2 * (8 * r + 4 * e + t);
          if (t0 >= ntok) vs[2 * r + e] &= 0xFF00u;
          if (t0 + 1 >= ntok) vs[2 * r + e] &= 0x00FFu;
        }
    }
    if (n_pv > 0 && !mbar_wait(pv_done, (n_pv - 1) & 1)) failed = true;  // V^T, P and O are free again
    tc_fence_after();
#pragma unroll
    for (int sg = 0; sg < 2; ++sg) {  // lane group sg: channels +2sg (lane g), +2sg+1 (lane g+8)
      uint32_t v[32];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t sc = f16x2_from_e4m3x2(vs[2 * r + e]);
          const uint32_t c0 = sg == 0 ? f16x2_from_e2m1_byte<0>(vw[2 * r + e]) : f16x2_from_e2m1_byte<2>(vw[2 * r + e]);
          const uint32_t c1 = sg == 0 ? f16x2_from_e2m1_byte<1>(vw[2 * r + e]) : f16x2_from_e2m1_byte<3>(vw[2 * r + e]);
          v[4 * r + e] = hmul2_u32(c0, sc);
          v[4 * r + 2 + e] = hmul2_u32(c1, sc);
        }
      tmem_st_16x256b_x8(tw + ((uint32_t)(16 * sg) << 16) + kColV, v);
    }

    // ---- S back from TMEM (fragment layout: rows g, g+8 of each 16-token group, columns 2t, 2t+1)
    if (!mbar_wait(s_full, (n_qk - 1) & 1)) failed = true;
    tc_fence_after();
    float S[2][4];
    tmem_ld_16x256b_x1(tw + kColS, S[0]);
    tmem_ld_16x256b_x1(tw + (16u << 16) + kColS, S[1]);
    tmem_wait_ld_only();
    if (ntok < kChunk) {
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        const int t0 = 32 * w + 16 * sl + g;
        if (t0 >= ntok) S[sl][0] = S[sl][1] = -INFINITY;
        if (t0 + 8 >= ntok) S[sl][2] = S[sl][3] = -INFINITY;
      }
    }
    float m0 = fmaxf(fmaxf(S[0][0], S[0][2]), fmaxf(S[1][0], S[1][2])) * st.cs[0];
    float m1 = fmaxf(fmaxf(S[0][1], S[0][3]), fmaxf(S[1][1], S[1][3])) * st.cs[1];
    // one reduction decides both the (rare) raise of the max and a failed wait
    if (wg_bar_or(idB, failed || m0 > st.m[0] + kLazySlack || m1 > st.m[1] + kLazySlack)) {
      if (wg_bar_or(idA, failed)) {
        failed = true;
        break;
      }
      // raise the running max to this stage's, for every row, in every thread
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, off));
        m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, off));
      }
      if (g == 0) {
        red_max[w * 8 + 2 * t] = m0;
        red_max[w * 8 + 2 * t + 1] = m1;
      }
      wg_bar(idA);
      float al[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float nm = fmaxf(fmaxf(st.mall[r], fmaxf(red_max[r], red_max[8 + r])), fmaxf(red_max[16 + r], red_max[24 + r]));
        al[r] = st.mall[r] == -INFINITY ? 0.0f : fast_exp2(st.mall[r] - nm);
        st.mall[r] = nm;
      }
      // this thread's rows 2t, 2t+1
      float a0 = al[0], a1 = al[1];
#pragma unroll
      for (int tt = 1; tt < 4; ++tt)
        if (t == tt) {
          a0 = al[2 * tt];
          a1 = al[2 * tt + 1];
        }
      float n0 = st.mall[0], n1 = st.mall[1];
#pragma unroll
      for (int tt = 1; tt < 4; ++tt)
        if (t == tt) {
          n0 = st.mall[2 * tt];
          n1 = st.mall[2 * tt + 1];
        }
      st.l[0] *= a0;
      st.l[1] *= a1;
      st.m[0] = n0;
      st.m[1] = n1;
      if (!first_pv) {  // O (its last update complete: pv_done waited above) times al, per row
        float o[8];
        tmem_ld_32x32b_x8(tw + kColO, o);
        tmem_wait_ld_only();
#pragma unroll
        for (int r = 0; r < 8; ++r) o[r] *= al[r];
        tmem_st_32x32b_x8(tw + kColO, o);
      }
    }
    const float nref0 = st.m[0] == -INFINITY ? 0.0f : -st.m[0];
    const float nref1 = st.m[1] == -INFINITY ? 0.0f : -st.m[1];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) {
      const float p0 = fast_exp2(fmaf(S[sl][0], st.cs[0], nref0));
      const float p1 = fast_exp2(fmaf(S[sl][1], st.cs[1], nref1));
      const float p2 = fast_exp2(fmaf(S[sl][2], st.cs[0], nref0));
      const float p3 = fast_exp2(fmaf(S[sl][3], st.cs[1], nref1));
      st.l[0] += p0 + p2;
      st.l[1] += p1 + p3;
      // P^T fragments: row g = query row, tokens 2t, 2t+1 (then +8) of this
      // 16-token group; their K index in the P tile follows the V^T columns
      const uint32_t pa = movmatrix_trans(pack_f16x2(p0, p1));
      const uint32_t pb = movmatrix_trans(pack_f16x2(p2, p3));
      const uint32_t kk = (uint32_t)(16 * (2 * w + sl) + 4 * t);
      const uint32_t off = pbuf + core_offset((uint32_t)g, kk, kTN);
      asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(off), "r"(pa) : "memory");
      asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(off + 4), "r"(pb) : "memory");
    }
    fence_async_smem();
    tmem_wait_st();
    tc_fence_before();
    if (wg_bar_or(idA, failed)) {
      failed = true;
      break;
    }
    if (i == 0) {  // O^T += V^T P^T
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kChunk / 16; ++ks)
        tc_mma_f16_ta(tmem_wg + kColO, tmem_wg + kColV + 8 * ks, pdesc + (uint64_t)(ks * 2 * (kTN / 8) * 8), kIdesc,
                      !first_pv || ks > 0);
      tc_commit(pv_done);
    }
    ++n_pv;
    first_pv = false;
    ++it;
    if (++sidx == kTStages) {
      sidx = 0;
      sphase ^= 1u;
    }
  }
  // `failed` is the same in every thread here: the loop ends on its count or
  // on a barrier reduction of it (then every thread set it)
  if (!failed && have) {
    flush();
    failed = wg_bar_or(idA, failed);  // the flush's own wait
  }
  if (failed) {
    if (i == 0) {
      set_flag(p.flag, KVQ_FLAG_TIMEOUT);
      *abort = 1;  // the producer stops issuing copies
      // the warpgroup's MMAs still running finish before the TMEM is freed
      if (n_qk > 0) mbar_wait(s_full, (n_qk - 1) & 1);
      if (n_pv > 0) mbar_wait(pv_done, (n_pv - 1) & 1);
    }
  }
}

template <int GT>
__global__ void __launch_bounds__(kTThreads, 1) decode_tc_kernel(const DecodeParams p) {
  extern __shared__ uint8_t tsm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp >= 4 * kTWG;
  const int wg = producer ? warp - 4 * kTWG : warp >> 2;
  uint8_t* wb = base + wg * TcWG::kBytes;
  const uint32_t wsb = sbase + (uint32_t)(wg * TcWG::kBytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kTWG * TcWG::kBytes);
  if (threadIdx.x < kTWG) {  // thread w: pipeline w's barriers and flags
    uint8_t* b = base + threadIdx.x * TcWG::kBytes;
    const uint32_t bs = sbase + (uint32_t)(threadIdx.x * TcWG::kBytes) + TcWG::kBar;
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(bs + 8 * s, 1);
      mbar_init(bs + 8 * (kTStages + s), 128);
    }
    mbar_init(bs + 8 * (2 * kTStages), 1);
    mbar_init(bs + 8 * (2 * kTStages + 1), 1);
    *reinterpret_cast<int*>(b + TcWG::kAbort) = 0;
    fence_barrier_init();
  }
  // the query and P tiles start zeroed (rows 8..15 are never written)
  for (int x = threadIdx.x; x < kTWG * 2 * kTOpBytes / 16; x += kTThreads) {
    const int pw = x / (2 * kTOpBytes / 16), r = x % (2 * kTOpBytes / 16);
    sts128(sbase + (uint32_t)(pw * TcWG::kBytes + TcWG::kQ + 16 * r), make_uint4(0u, 0u, 0u, 0u));
  }
  fence_async_smem();
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  const int vidx = blockIdx.x * kTWG + wg, vcount = gridDim.x * kTWG;
  int64_t total, v0, v1;
  Walker wk;
  plan(p, vidx, vcount, total, v0, v1, wk);
  if (v0 < v1) {
    if (producer) {
      if (lane == 0) tc_producer<GT>(p, wb, wsb, wk, v1);
    } else {
      tc_consumer<GT>(p, wb, wsb, tmem + (uint32_t)wg * kColsPerWG, wg, wk, v1, total, vidx, vcount);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTTmemCols);
}

template <int GT>
kvq_status launch_decode_tc_g(const DecodeParams& dp, cudaStream_t s) {
  static DeviceOnce attr_set;  // the shared-memory opt-in, once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(decode_tc_kernel<GT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmemBytes) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  const int sms = device_sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  decode_tc_kernel<GT><<<sms, kTThreads, kTSmemBytes, s>>>(dp);
  return launch_status();
}

}  // namespace

// head_dim 128 decode on the tensor cores; the grid is one CTA per SM with
// three pipelines each, so the ranges and partial slots are those of
// 3 x (number of SMs) CTAs of the mma.sync kernel.
kvq_status launch_decode_tc(const DecodeParams& dp, cudaStream_t s) {
  switch (dp.page < kChunk ? dp.page : kChunk) {
    case 16: return launch_decode_tc_g<16>(dp, s);
    case 32: return launch_decode_tc_g<32>(dp, s);
    case 64: return launch_decode_tc_g<64>(dp, s);
    default: return launch_decode_tc_g<kChunk>(dp, s);
  }
}

}  // namespace kvq
