// kvq_prefill.cu -- chunked-prefill attention over the FP4 (or NVFP4) paged
// cache on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Method: "Quantising the KV cache", section "Code" -- the quantised K and V
// feed an unchanged attention -- applied to a chunk of new query tokens whose
// keys and values are already in the cache: query token i of a chunk of C in
// a sequence of T cached positions sits at position T - C + i and attends
// positions 0..T - C + i (causal), all read from the FP4 cache.  With many
// query rows per cache tile the products are dense (unlike decode), so they
// run on the tensor cores; the cache is dequantised once per tile into shared
// memory and shared by the CTA's 256 query rows.
//
// CTA = the G query heads of one kv head times 256/G consecutive query tokens
// of one sequence: 256 query rows as two 128-row query tiles (A and B) that
// share each dequantised cache tile.  Fourteen warps in four roles run as a
// pipeline over the sequence's 128-position cache tiles:
//   softmax (2 x 4 warps)  warpgroup X serves query tile X, thread r owns row
//                       r: per 64-score half of the tile, read from TMEM once,
//                       the half's max against the lazy reference (raised only
//                       past +8 in the log2 domain; O rescaled in TMEM then),
//                       then P = 2^(S - m) as f16 pairs written back over the
//                       first half of S_X's columns; the causal mask only on
//                       the diagonal tiles
//   dequant (4 warps)   K^ [128 pos][d] (one slot) and V^ [d][128 pos] (two
//                       slots) into shared memory in the tensor core's
//                       K-major core-matrix layout (f16, E2M1 code times E4M3
//                       scale; positions past the end 0)
//   loader (1 thread)   bulk copies of the FP4 tiles, 3 in flight
//   MMA (1 thread)      S_X(j) = Q_X K^(j)^T   tcgen05.mma M=128 N=128 K=d
//                       O_X += P_X(j) V^(j)   tcgen05.mma M=128 N=d K=128, P_X
//                                           read from TMEM, O_X in TMEM
//                       in the order O_A(j), S_A(j+1), O_B(j), S_B(j+1)
// mbarriers hand each buffer from producer to consumer and back (MMA
// completions arrive via tcgen05.commit).  V^ has two slots so that the
// dequantisation of tile j+1's V^ never waits for tile j's last PV product:
// with one slot that dequantisation sat between O_B(j) and O_A(j+1) on every
// tile (2.10 -> 1.78 ms on prefill_attn); K^'s single slot is refilled while
// the softmax of tile j runs.  Finally O / l (times the NVFP4 value scale)
// goes to global memory.  Every wait is bounded; a timeout raises the CTA's
// abort word, every role leaves its loop, copies and MMAs still in flight are
// waited for (bounded), the TMEM is freed and the timeout flag set.
#include "kvq_common.cuh"
#include "kvq_host.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kPTile = 128;     // cache positions per tile
constexpr int kPRows = 128;     // rows of one query tile (the MMA's M)
constexpr int kQTiles = 2;      // query tiles per CTA, sharing each dequantised K^/V^ tile
constexpr int kCtaRows = kQTiles * kPRows;
constexpr int kSoftWarps = 4 * kQTiles;  // warps 0-7: softmax, warpgroup X = query tile X, thread = row
constexpr int kDeqWarps = 4;    // warps 8-11: FP4 -> f16 dequantisation of K^ and V^
constexpr int kLoadWarp = kSoftWarps + kDeqWarps;  // lane 0: bulk copies of the FP4 tiles
constexpr int kMmaWarp = kLoadWarp + 1;            // lane 0: tensor-core issue
constexpr int kPThreads = 32 * (kMmaWarp + 1);
constexpr int kOCol = kQTiles * kPTile;  // TMEM: S_X (then P_X) at [128 X, +128), O_X at [256 + 128 X, +d)
constexpr int kTmemCols = 512;
constexpr int kFp4Stages = 3;   // FP4 tiles in flight
constexpr int kKSlots = 1;      // K^ slots (refilled while the softmax runs)
constexpr int kVSlots = 2;      // V^ slots (see above)
constexpr float kPSlack = 8.0f;
constexpr uint32_t kPollNs = 20000;  // suspend hint of a barrier poll

// mbarriers, by index
enum : int {
  kBFp4Full = 0,                        // [kFp4Stages] tile landed (bulk-copy bytes)
  kBFp4Empty = kBFp4Full + kFp4Stages,  // [kFp4Stages] dequantisers done with the tile (128 arrivals)
  kBKFull = kBFp4Empty + kFp4Stages,    // [kKSlots] K^ slot written (128 arrivals)
  kBKEmpty = kBKFull + kKSlots,         // [kKSlots] both S = Q K^T done reading it (MMA commit)
  kBVFull = kBKEmpty + kKSlots,         // [kVSlots] V^ slot written (128 arrivals)
  kBVEmpty = kBVFull + kVSlots,         // [kVSlots] both O += P V done reading it (MMA commit)
  kBSFull = kBVEmpty + kVSlots,         // [kQTiles] S_X in TMEM
  kBPFull = kBSFull + kQTiles,          // [kQTiles] P_X in TMEM, O_X rescaled (128 arrivals)
  kBPvDone = kBPFull + kQTiles,         // [kQTiles] O_X += P_X V done (S_X's TMEM free again)
  kNumBars = kBPvDone + kQTiles
};

struct PrefillParams {
  const int32_t* lens;
  const int32_t* page_table;
  const uint8_t* pool;
  const uint16_t* q;
  float* out;
  int32_t* flag;
  const float* k_gscale;  // NVFP4 second-level scales [Hkv] (nullptr: FP4)
  const float* v_gscale;
  int64_t num_pages;
  int32_t batch, hkv, g, hq, page, max_pages, chunk;
  float qk_log2;
};

template <int D>
struct PGeo {
  static constexpr int kTileBytes = kPTile * 9 * D / 8;   // FP4 bytes of 128 positions of one kv head
  static constexpr int kOpBytes = kPTile * D * 2;         // one query tile, K^ slot or V^ (f16, core layout)
  static constexpr int kQ = 0;                            // Q  [kQTiles][128 rows][D]
  static constexpr int kK = kQ + kQTiles * kOpBytes;      // K^ [kKSlots][128 positions][D]
  static constexpr int kV = kK + kKSlots * kOpBytes;      // V^ [kVSlots][D channels][128 positions]
  static constexpr int kStage = kV + kVSlots * kOpBytes;  // FP4 tiles [kFp4Stages]
  static constexpr int kBars = kStage + kFp4Stages * kTileBytes;
  static constexpr int kUsed = kBars + 8 * kNumBars + 8 + 128;  // + TMEM slot, abort word, alignment slack
  // at least half an SM's shared memory, so that one CTA (holding all 512
  // TMEM columns) runs per SM
  static constexpr int kBytes = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static_assert(kTileBytes % 16 == 0 && kStage % 128 == 0 && kBars % 16 == 0, "shared-memory layout alignment");
  static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
};

// Bounded wait on an mbarrier phase that also gives up once another role has
// given up; the first to time out raises the CTA's abort word.
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, kPollNs)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
}

// pwait with one outcome for the whole warp (TMEM accesses are warp-collective).
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xFFFFFFFFu, pwait(bar, parity, abort));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Packed pairs of fp32 (low word first) and their one-instruction arithmetic.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Issue the bulk copies of tile j (its groups that start before position T)
// into a stage buffer, arming `bar` with their byte count.
template <int D, int GT>
__device__ void issue_tile(const PrefillParams& p, int b, int h, int j, int T, uint32_t dst, uint32_t bar) {
  constexpr int kGroupBytes = GT * 9 * D / 8;
  constexpr int kGroups = kPTile / GT;
  uint32_t bytes = 0;
  int64_t src[kGroups];
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    src[gi] = -1;
    const int64_t pos = (int64_t)j * kPTile + gi * GT;
    if (pos >= T) continue;
    const int64_t pg = pos / p.page;
    const int slot = (int)(pos % p.page);
    if (pg >= p.max_pages) {
      set_flag(p.flag, KVQ_FLAG_PAGE_OOB);
      continue;
    }
    const int64_t phys = p.page_table ? (int64_t)__ldg(p.page_table + (int64_t)b * p.max_pages + pg)
                                      : (int64_t)b * p.max_pages + pg;
    if (phys < 0 || phys >= p.num_pages) {
      set_flag(p.flag, KVQ_FLAG_PAGE_OOB);
      continue;
    }
    src[gi] = ((phys * p.hkv + h) * (p.page / GT) + slot / GT) * kGroupBytes;
    bytes += kGroupBytes;
  }
  mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi)
    if (src[gi] >= 0) bulk_g2s(dst + gi * kGroupBytes, p.pool + src[gi], kGroupBytes, bar);
}

// K^ of one staged tile into its operand layout ([position][channel],
// K-major); positions >= valid (past the sequence end) are written as 0.
// Thread n (of 128) takes position n, one 32-channel quarter per step: a
// 16-byte code load, the quarter's two block scales, four 16-byte stores.  The
// quarter order is rotated by position so that the 8 lanes of a load phase
// (8 consecutive positions, D/2 bytes apart) hit 8 different bank groups.
template <int D, int GT>
__device__ __forceinline__ void dequant_k(uint32_t stage, uint32_t kdst, int valid, int n) {
  constexpr int NB = D / 16;
  constexpr int kGroupBytes = GT * 9 * D / 8;
  constexpr int kQuarters = D / 32;
  constexpr int kRotShift = D == 128 ? 1 : 2;  // log2(positions per 128 code bytes)
  const uint32_t grp = stage + (uint32_t)((n / GT) * kGroupBytes);
  const int ln = n % GT;
#pragma unroll 2
  for (int m = 0; m < kQuarters; ++m) {
    const int qq = (m + (n >> kRotShift)) & (kQuarters - 1);
    uint32_t r[16];
    if (n < valid) {
      const uint4 w = lds128(grp + (uint32_t)(ln * (D / 2) + qq * 16));
      const uint32_t s2 = f16x2_from_e4m3x2(lds16(grp + (uint32_t)(GT * (D / 2) + ln * NB + 2 * qq)));
      const uint32_t sA = prmt(s2, 0u, 0x1010u), sB = prmt(s2, 0u, 0x3232u);  // each block's scale, twice
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t t[4];
        f16x2x4_from_e2m1x8(ws[k], t);
#pragma unroll
        for (int i = 0; i < 4; ++i) r[4 * k + i] = hmul2_u32(t[i], k < 2 ? sA : sB);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = 0u;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      sts128(kdst + core_offset((uint32_t)n, (uint32_t)(qq * 32 + 8 * k), kPTile),
             make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]));
  }
}

// V^ of one staged tile into its operand layout ([channel][position],
// K-major over positions).  Item (8 channels c..c+7, 8 positions = 4
// token-pair rows): an 8-byte code load per pair row (each byte pairs the
// row's two positions; the 8 channels share one 16-channel block scale), the
// pair's scales, one 16-byte store per channel.
template <int D, int GT>
__device__ __forceinline__ void dequant_v(uint32_t stage, uint32_t vdst, int valid, int dt) {
  constexpr int NB = D / 16;
  constexpr int kGroupBytes = GT * 9 * D / 8;
#pragma unroll 1
  for (int it = dt; it < (D / 8) * (kPTile / 8); it += 32 * kDeqWarps) {
    const int c = (it % (D / 8)) * 8;
    const int n0 = (it / (D / 8)) * 8;
    const int i0 = (n0 % GT) >> 1;  // first pair row, a multiple of 4
    const uint32_t grp = stage + (uint32_t)((n0 / GT) * kGroupBytes);
    const uint32_t codes = grp + (uint32_t)(GT * (D / 2 + NB) + i0 * D);  // pair row i0
    const uint32_t scales = grp + (uint32_t)(GT * (D + NB) + i0 * 2 * NB + 2 * (c >> 4));
    // the 8 lanes of a store phase write channels 8t + k: rotating each
    // thread's bytes by r = (c / 8) mod 8 spreads them over 8 bank groups
    const uint32_t r = (uint32_t)(c >> 3) & 7u;
    const uint32_t sh = 8u * (r & 3u);
    uint32_t res[8][4];  // [rotated channel][pair]
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + 2 * q;  // even position of the pair
      uint32_t t[2][4];
      uint32_t sc = 0u;
      uint2 w = make_uint2(0u, 0u);
      if (n < valid) {
        // pair row i0 + q (i0 % 4 == 0): channel chunks permuted by the row index
        const int phys = (D == 64) ? 8 * ((c >> 3) ^ (((q >> 1) & 1) << 2)) : 16 * ((c >> 4) ^ (q << 1)) + (c & 15);
        w = lds64(codes + (uint32_t)(q * D + phys));
        uint32_t s2 = lds16(scales + (uint32_t)(q * 2 * NB));
        if (n + 1 >= valid) s2 &= 0x00FFu;  // the pair's second position is past the end: scale 0
        sc = f16x2_from_e4m3x2(s2);
      }
      const uint32_t a = (r & 4u) ? w.y : w.x, bb = (r & 4u) ? w.x : w.y;
      f16x2x4_from_e2m1x8(__funnelshift_r(a, bb, sh), t[0]);  // byte k -> channel c + (k + r) % 8
      f16x2x4_from_e2m1x8(__funnelshift_r(bb, a, sh), t[1]);
#pragma unroll
      for (int k = 0; k < 8; ++k) res[k][q] = hmul2_u32(t[k >> 2][k & 3], sc);
    }
    const uint32_t row0 = vdst + core_offset((uint32_t)c, (uint32_t)n0, D);  // channel c; c % 8 == 0
#pragma unroll
    for (int k = 0; k < 8; ++k)
      sts128(row0 + (((uint32_t)k + r) & 7u) * 16u, make_uint4(res[k][0], res[k][1], res[k][2], res[k][3]));
  }
}

// Row max of 32 raw scores of a tile (positions >= lim masked unless FAST),
// into four independent running maxima.
template <bool FAST>
__device__ __forceinline__ void chunk_max(const uint32_t (&v)[32], int c0, int lim, float (&m)[4]) {
  if (FAST) {
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i & 3] = fmax3(m[i & 3], __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i < lim) m[i & 3] = fmaxf(m[i & 3], __uint_as_float(v[i]));
  }
}

// P = 2^(S * cs - m) for 32 scores, as 16 f16 pairs; the row sum goes into
// two packed running sums.  Positions >= lim are masked unless FAST.
template <bool FAST>
__device__ __forceinline__ void chunk_p(const uint32_t (&v)[32], uint32_t* w, int c0, int lim, uint64_t cs2,
                                        uint64_t nref2, uint64_t (&l2)[2]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float y0, y1;
    f2unpack(ffma2(f2pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), cs2, nref2), y0, y1);
    float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
    if (!FAST) {
      if (c0 + 2 * i >= lim) e0 = 0.0f;
      if (c0 + 2 * i + 1 >= lim) e1 = 0.0f;
    }
    l2[i & 1] = fadd2(l2[i & 1], f2pack(e0, e1));
    w[i] = pack_f16x2(e0, e1);
  }
}

template <int D, int GT>
__global__ void __launch_bounds__(kPThreads, 1) prefill_fp4_kernel(const PrefillParams p) {
  using G = PGeo<D>;
  extern __shared__ uint8_t psm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(psm_raw) + 127) & ~uintptr_t(127));
  const uint32_t sb = smem_addr(base);
  const uint32_t bars = sb + G::kBars;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + G::kBars + 8 * kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qpb = kCtaRows / p.g;  // query tokens per CTA
  const int nqb = (p.chunk + qpb - 1) / qpb;
  const int qb = (int)(blockIdx.x % nqb);
  const int bh = (int)(blockIdx.x / nqb);
  const int h = bh % p.hkv, b = bh / p.hkv;
  const int32_t T = __ldg(p.lens + b);
  // softmax threads: CTA row tid = query token ti of the chunk, query head hh;
  // query tile X = tid / 128, row tid % 128 of it
  const int ti = qb * qpb + tid / p.g;
  const int hh = h * p.g + tid % p.g;
  const int X = tid / kPRows;
  const bool row_ok = tid < kCtaRows && ti < p.chunk;
  float* orow = p.out + (((int64_t)b * p.chunk + ti) * p.hq + hh) * D;
  if (T < p.chunk) {  // the chunk's own tokens must be in the cache
    if (tid == 0) set_flag(p.flag, KVQ_FLAG_BAD_LENGTH);
    if (row_ok)
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t pos_r = (int64_t)T - p.chunk + ti;          // last position this row attends
  const int64_t pos_min = (int64_t)T - p.chunk + qb * qpb;  // ... the CTA's first query token
  const int last_ti = min(p.chunk, (qb + 1) * qpb) - 1;
  const int ntiles = (int)(((int64_t)T - p.chunk + last_ti) / kPTile) + 1;

  if (tid == 0) {
    for (int i = 0; i < kFp4Stages; ++i) {
      mbar_init(bars + 8 * (kBFp4Full + i), 1);
      mbar_init(bars + 8 * (kBFp4Empty + i), 32 * kDeqWarps);
    }
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(bars + 8 * (kBKFull + i), 32 * kDeqWarps);
      mbar_init(bars + 8 * (kBKEmpty + i), 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bars + 8 * (kBVFull + i), 32 * kDeqWarps);
      mbar_init(bars + 8 * (kBVEmpty + i), 1);
    }
    for (int i = 0; i < kQTiles; ++i) {
      mbar_init(bars + 8 * (kBSFull + i), 1);
      mbar_init(bars + 8 * (kBPFull + i), 32 * 4);
      mbar_init(bars + 8 * (kBPvDone + i), 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);

  // query row -> f16 with a power-of-two prescale (exact for bf16 values in
  // range), into the A-operand layout of its query tile; the factor returns in
  // the score scale
  float cs = 0.0f;
  if (warp < kSoftWarps) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (((int64_t)b * p.chunk + ti) * p.hq + hh) * D);
    uint32_t amax_bits = 0u;  // |x| of the row's largest element (bf16 bits, upper half)
    if (row_ok) {
#pragma unroll 4
      for (int i = 0; i < D / 8; ++i) {
        const uint4 w = __ldg(src + i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          amax_bits = max(amax_bits, max((ws[k] << 16) & 0x7FFF0000u, ws[k] & 0x7FFF0000u));
      }
    }
    const float amax = __uint_as_float(amax_bits);
    int k = 0;
    if (amax > 0.0f && amax <= 3.4e38f) {
      const int e = (int)((amax_bits >> 23) & 0xFF) - 127;
      k = min(100, max(-113, 14 - e));
    }
    const float up = __uint_as_float((uint32_t)(k + 127) << 23);
    const uint32_t qdst = sb + G::kQ + X * G::kOpBytes;
#pragma unroll 4
    for (int c8 = 0; c8 < D / 8; ++c8) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok) w = __ldg(src + c8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = pack_f16x2(bf16_lo(ws[j]) * up, bf16_hi(ws[j]) * up);
      sts128(qdst + core_offset((uint32_t)(tid % kPRows), (uint32_t)(c8 * 8), kPRows),
             make_uint4(f[0], f[1], f[2], f[3]));
    }
    const float sk = p.k_gscale ? __ldg(p.k_gscale + h) : 1.0f;
    cs = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - k) << 23);
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp < kSoftWarps) {
    // ---------------------------------------------------------------- softmax
    // this warp's 32 TMEM lanes (rows), in query tile X's S/P and O columns
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t sp = t_lane + (uint32_t)(X * kPTile);
    const uint32_t op = t_lane + (uint32_t)(kOCol + X * kPTile);
    const uint32_t s_full = bars + 8 * (kBSFull + X), p_full = bars + 8 * (kBPFull + X);
    const uint32_t pv_done = bars + 8 * (kBPvDone + X);
    const uint64_t cs2 = f2pack(cs, cs);
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      if (!(ok = wwait(s_full, (uint32_t)j & 1u, abort))) break;
      tc_fence_after();
      const int64_t p0 = (int64_t)j * kPTile;
      const bool fast = p0 + kPTile - 1 <= pos_min;  // no position of the tile masked for any row
      const int lim = row_ok ? (int)min((int64_t)kPTile, max((int64_t)0, pos_r - p0 + 1)) : 0;
      // the tile in two halves of 64 scores, each read from TMEM once: its
      // max (raw scores; cs > 0) against the lazy reference, then its P over
      // scores already held in registers (half h -> columns [32h, 32h + 32)).
      // A raise of the reference shrinks what was accumulated against the old
      // one: l, O and, for the second half, the first half's P.
      uint64_t l2[2] = {0ull, 0ull};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t va[32], vb[32];
        tmem_ld32_async(sp + (uint32_t)(64 * hf), va);
        tmem_ld32_async(sp + (uint32_t)(64 * hf + 32), vb);
        tmem_wait_ld(va);
        tmem_wait_ld(vb);
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (fast) {
          chunk_max<true>(va, 64 * hf, lim, m4);
          chunk_max<true>(vb, 64 * hf + 32, lim, m4);
        } else {
          chunk_max<false>(va, 64 * hf, lim, m4);
          chunk_max<false>(vb, 64 * hf + 32, lim, m4);
        }
        const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * cs;
        float al = 1.0f;
        if (mt > m_run + kPSlack) {
          if (m_run != -INFINITY) al = fast_exp2(m_run - mt);
          m_run = mt;
        }
        if (__any_sync(0xFFFFFFFFu, al != 1.0f)) {  // TMEM accesses are warp-collective
          if (hf == 1) {  // the first half's P, columns [0, 32)
            const uint32_t al2 = pack_f16x2(al, al);
            tmem_wait_st();
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint32_t pw[16];
              tmem_ld16(sp + (uint32_t)(16 * k), pw);
#pragma unroll
              for (int i = 0; i < 16; ++i) pw[i] = hmul2_u32(pw[i], al2);
              tmem_st16_async(sp + (uint32_t)(16 * k), pw);
            }
          }
          {
            float a0, a1, b0, b1;
            f2unpack(l2[0], a0, a1);
            f2unpack(l2[1], b0, b1);
            l2[0] = f2pack(a0 * al, a1 * al);
            l2[1] = f2pack(b0 * al, b1 * al);
          }
          if (j > 0) {  // O: once O_X += P_X V of the previous tile is done
            if (!(ok = wwait(pv_done, (uint32_t)(j - 1) & 1u, abort))) break;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
              uint32_t o[16];
              tmem_ld16(op + (uint32_t)c0, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
              tmem_st16_async(op + (uint32_t)c0, o);
            }
          }
        }
        l_run *= al;
        const float nref = m_run == -INFINITY ? 0.0f : -m_run;
        const uint64_t nref2 = f2pack(nref, nref);
        uint32_t w[16];
        if (fast) {
          chunk_p<true>(va, w, 64 * hf, lim, cs2, nref2, l2);
          tmem_st16_async(sp + (uint32_t)(32 * hf), w);
          chunk_p<true>(vb, w, 64 * hf + 32, lim, cs2, nref2, l2);
          tmem_st16_async(sp + (uint32_t)(32 * hf + 16), w);
        } else {
          chunk_p<false>(va, w, 64 * hf, lim, cs2, nref2, l2);
          tmem_st16_async(sp + (uint32_t)(32 * hf), w);
          chunk_p<false>(vb, w, 64 * hf + 32, lim, cs2, nref2, l2);
          tmem_st16_async(sp + (uint32_t)(32 * hf + 16), w);
        }
      }
      if (!ok) break;
      tmem_wait_st();
      {
        float a0, a1, b0, b1;
        f2unpack(l2[0], a0, a1);
        f2unpack(l2[1], b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
      }
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // O / l (times the NVFP4 value scale) once the last O_X += P_X V is done
    if (ok) ok = wwait(pv_done, (uint32_t)(ntiles - 1) & 1u, abort);
    if (ok) {
      tc_fence_after();
      const float vs = p.v_gscale ? __ldg(p.v_gscale + h) : 1.0f;
      const float inv = l_run > 0.0f ? vs / l_run : 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(op + (uint32_t)c0, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(orow + c0 + i) =
                make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                            __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
        }
      }
    }
  } else if (warp < kSoftWarps + kDeqWarps) {
    // ---------------------------------------------------------- dequantisation
    const int dt = tid - 32 * kSoftWarps;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kFp4Stages, slot = j % kKSlots;
      const uint32_t stage = sb + G::kStage + s * G::kTileBytes;
      const int valid = (int)min((int64_t)kPTile, (int64_t)T - (int64_t)j * kPTile);
      if (!wwait(bars + 8 * (kBFp4Full + s), (uint32_t)(j / kFp4Stages) & 1u, abort)) break;
      if (j >= kKSlots && !wwait(bars + 8 * (kBKEmpty + slot), (uint32_t)(j / kKSlots - 1) & 1u, abort)) break;
      dequant_k<D, GT>(stage, sb + G::kK + slot * G::kOpBytes, valid, dt);
      fence_async_smem();
      mbar_arrive(bars + 8 * (kBKFull + slot));
      const int vslot = j % kVSlots;
      if (j >= kVSlots && !wwait(bars + 8 * (kBVEmpty + vslot), (uint32_t)(j / kVSlots - 1) & 1u, abort)) break;
      dequant_v<D, GT>(stage, sb + G::kV + vslot * G::kOpBytes, valid, dt);
      mbar_arrive(bars + 8 * (kBFp4Empty + s));
      fence_async_smem();
      mbar_arrive(bars + 8 * (kBVFull + vslot));
    }
  } else if (warp == kLoadWarp) {
    // ---------------------------------------------------------- bulk copies
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % kFp4Stages;
        if (j >= kFp4Stages && !pwait(bars + 8 * (kBFp4Empty + s), (uint32_t)(j / kFp4Stages - 1) & 1u, abort))
          break;
        issue_tile<D, GT>(p, b, h, j, T, sb + G::kStage + s * G::kTileBytes, bars + 8 * (kBFp4Full + s));
        issued = j + 1;
      }
      if (*abort) {  // let copies still in flight land before the shared memory goes away
        for (int j = max(0, issued - kFp4Stages); j < issued; ++j) {
          const uint32_t bar = bars + 8 * (kBFp4Full + j % kFp4Stages);
          const uint32_t par = (uint32_t)(j / kFp4Stages) & 1u;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait_hint(bar, par, kPollNs) && global_ns() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (lane == 0) {
    // ---------------------------------------------------------- tensor cores
    // order: S_A(0), S_B(0), then per tile j: O_A += P_A V^(j), S_A(j+1),
    // O_B += P_B V^(j), S_B(j+1) -- each query tile's next scores follow its
    // own O update (P_X lives in S_X's columns, so S_X(j+1) waits for that
    // update to complete) and never wait for the other tile's softmax
    constexpr uint32_t kIdS = idesc_f16_f32(kPRows, kPTile);
    constexpr uint32_t kIdO = idesc_f16_f32(kPRows, D);
    uint32_t last_bar = 0, last_par = 0;
    auto issue_s = [&](int jj, int x) {
      const uint64_t dq = smem_desc(sb + G::kQ + x * G::kOpBytes, (kPRows / 8) * 128, 128);
      const uint64_t dk = smem_desc(sb + G::kK + (jj % kKSlots) * G::kOpBytes, (kPTile / 8) * 128, 128);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc_mma_f16(tmem + (uint32_t)(x * kPTile), dq + (uint64_t)(ks * 2 * (kPRows / 8) * 8),
                   dk + (uint64_t)(ks * 2 * (kPTile / 8) * 8), kIdS, ks > 0);
      tc_commit(bars + 8 * (kBSFull + x));
      last_bar = bars + 8 * (kBSFull + x);
      last_par = (uint32_t)jj & 1u;
    };
    bool ok = pwait(bars + 8 * kBKFull, 0u, abort);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      issue_s(0, 1);
      tc_commit(bars + 8 * kBKEmpty);
    }
    for (int j = 0; j < ntiles && ok; ++j) {
      if (!(ok = pwait(bars + 8 * (kBVFull + j % kVSlots), (uint32_t)(j / kVSlots) & 1u, abort))) break;
#pragma unroll
      for (int x = 0; x < kQTiles; ++x) {
        if (!(ok = pwait(bars + 8 * (kBPFull + x), (uint32_t)j & 1u, abort))) break;
        tc_fence_after();
        const uint64_t dv = smem_desc(sb + G::kV + (j % kVSlots) * G::kOpBytes, (D / 8) * 128, 128);
#pragma unroll
        for (int ks = 0; ks < kPTile / 16; ++ks)
          tc_mma_f16_ta(tmem + (uint32_t)(kOCol + x * kPTile), tmem + (uint32_t)(x * kPTile + ks * 8),
                        dv + (uint64_t)(ks * 2 * (D / 8) * 8), kIdO, j > 0 || ks > 0);
        tc_commit(bars + 8 * (kBPvDone + x));
        last_bar = bars + 8 * (kBPvDone + x);
        last_par = (uint32_t)j & 1u;
        if (x == kQTiles - 1) tc_commit(bars + 8 * (kBVEmpty + j % kVSlots));
        if (j + 1 < ntiles) {
          const int jn = j + 1;
          if (x == 0 && !(ok = pwait(bars + 8 * (kBKFull + jn % kKSlots), (uint32_t)(jn / kKSlots) & 1u, abort)))
            break;
          if (!(ok = pwait(bars + 8 * (kBPvDone + x), (uint32_t)j & 1u, abort))) break;
          tc_fence_after();
          issue_s(jn, x);
          if (x == kQTiles - 1) tc_commit(bars + 8 * (kBKEmpty + jn % kKSlots));
        }
      }
    }
    if (*abort && last_bar != 0) {  // MMAs still running when the CTA gave up: let them finish
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait_hint(last_bar, last_par, kPollNs) && global_ns() - t0 < 20000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && *abort) set_flag(p.flag, KVQ_FLAG_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

int prefill_smem_bytes(int d) { return d == 128 ? PGeo<128>::kBytes : PGeo<64>::kBytes; }

template <int D, int GT>
kvq_status launch_prefill_g(const PrefillParams& pp, cudaStream_t s, unsigned grid) {
  static DeviceOnce attr_set;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(prefill_fp4_kernel<D, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PGeo<D>::kBytes) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  prefill_fp4_kernel<D, GT><<<grid, kPThreads, PGeo<D>::kBytes, s>>>(pp);
  return launch_status();
}

template <int D>
kvq_status launch_prefill(const PrefillParams& pp, cudaStream_t s, unsigned grid) {
  switch (pp.page < kPTile ? pp.page : kPTile) {
    case 16: return launch_prefill_g<D, 16>(pp, s, grid);
    case 32: return launch_prefill_g<D, 32>(pp, s, grid);
    case 64: return launch_prefill_g<D, 64>(pp, s, grid);
    default: return launch_prefill_g<D, kPTile>(pp, s, grid);
  }
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_prefill_attn(const kvq_cache* cache, int32_t batch, int32_t num_q_heads, int32_t chunk,
                                       const int32_t* d_seq_lens, const void* q, float softmax_scale, float* out,
                                       int32_t* d_err_flag, kvq_stream stream) {
  if (batch < 1 || chunk < 1) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_status st = check_cache(cache, batch);
  if (st != KVQ_OK) return st;
  if (!is_fp4_layout(cache)) return KVQ_ERR_INVALID_ARGUMENT;
  const int hkv = cache->num_kv_heads, D = cache->head_dim;
  if (num_q_heads < hkv || num_q_heads % hkv != 0) return KVQ_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / hkv;
  if (!(softmax_scale > 0.0f) || !(softmax_scale < 3.0e38f)) return KVQ_ERR_INVALID_ARGUMENT;
  if (d_seq_lens == nullptr || q == nullptr || out == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(q, 16) || !aligned_to(out, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (g > 8 || (kCtaRows % g) != 0) return KVQ_ERR_UNSUPPORTED;
  const int64_t nqb = ((int64_t)chunk + kCtaRows / g - 1) / (kCtaRows / g);
  const int64_t grid = nqb * batch * hkv;
  if (grid > 0x7FFFFFFF) return KVQ_ERR_UNSUPPORTED;
  PrefillParams pp;
  pp.lens = d_seq_lens;
  pp.page_table = cache->page_table;
  pp.pool = static_cast<const uint8_t*>(cache->data);
  pp.q = static_cast<const uint16_t*>(q);
  pp.out = out;
  pp.flag = d_err_flag;
  const bool nv = cache->format == KVQ_FORMAT_NVFP4;
  pp.k_gscale = nv ? static_cast<const float*>(cache->k_scale) : nullptr;
  pp.v_gscale = nv ? static_cast<const float*>(cache->v_scale) : nullptr;
  pp.num_pages = cache->num_pages;
  pp.batch = batch;
  pp.hkv = hkv;
  pp.g = g;
  pp.hq = num_q_heads;
  pp.page = cache->page_size;
  pp.max_pages = cache->max_pages_per_seq;
  pp.chunk = chunk;
  pp.qk_log2 = softmax_scale * 1.4426950408889634f;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return D == 128 ? launch_prefill<128>(pp, s, (unsigned)grid) : launch_prefill<64>(pp, s, (unsigned)grid);
}
