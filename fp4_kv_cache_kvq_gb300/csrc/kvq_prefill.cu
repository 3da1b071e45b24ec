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
// memory and shared by the CTA's 128 query rows.
//
// CTA = 128 threads, one per query row: the G query heads of one kv head times
// 128/G consecutive query tokens of one sequence.  Per 128-position tile:
//   bulk copy of the tile's FP4 groups (double-buffered, thread 0)
//   dequantise K^ [128 pos][d] and V^ [d][128 pos] into shared memory in the
//     tensor core's K-major core-matrix layout (f16, E2M1 code times E4M3
//     scale; positions past the sequence end are zero)
//   S = Q K^T            tcgen05.mma M=128 N=128 K=d, into TMEM
//   online softmax, thread r owns row r: S from TMEM, scale, causal mask,
//     lazy max (raised only past +8 in the log2 domain; O rescaled in TMEM
//     then), P in f16 to shared memory
//   O += P V             tcgen05.mma M=128 N=d K=128, into TMEM
// Finally O / l (times the NVFP4 value scale) to global memory.  Every wait is
// bounded; a timeout sets a flag, and the CTA waits (bounded) for its copies,
// frees its TMEM and returns.
#include "kvq_common.cuh"
#include "kvq_host.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kPTile = 128;     // cache positions per tile
constexpr int kPRows = 128;     // query rows per CTA
constexpr int kPThreads = 128;  // one thread per row
constexpr int kTmemCols = 256;  // S: columns [0, 128), O: [128, 128 + d)
constexpr float kPSlack = 8.0f;

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
  static constexpr int kTileBytes = kPTile * 9 * D / 8;  // FP4 bytes of 128 positions of one kv head
  static constexpr int kQ = 0;                           // Q  [128 rows][D]        f16, core layout
  static constexpr int kK = kQ + kPRows * D * 2;         // K^ [128 positions][D]
  static constexpr int kV = kK + kPTile * D * 2;         // V^ [D channels][128 positions]
  static constexpr int kP = kV + D * kPTile * 2;         // P  [128 rows][128 positions]
  static constexpr int kStage = kP + kPRows * kPTile * 2;
  static constexpr int kBars = kStage + 2 * kTileBytes;  // full[2], mma, tmem slot, abort
  static constexpr int kBytes = kBars + 64 + 128;        // + alignment slack
  static_assert(kTileBytes % 16 == 0 && kStage % 128 == 0 && kBars % 16 == 0, "shared-memory layout alignment");
};

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

// K^ and V^ of one staged tile into the operand layouts; positions >= valid
// (past the sequence end) are written as 0.
template <int D, int GT>
__device__ __forceinline__ void dequant_tile(uint32_t stage, uint32_t kdst, uint32_t vdst, int valid) {
  constexpr int NB = D / 16;
  constexpr int kGroupBytes = GT * 9 * D / 8;
  const int tid = threadIdx.x;
  // K^: thread n takes position n, one 32-channel quarter per step: a 16-byte
  // code load, the quarter's two block scales, four 16-byte stores.  The
  // quarter order is rotated by position so that the 8 lanes of a load phase
  // (8 consecutive positions, D/2 bytes apart) hit 8 different bank groups.
  static_assert(kPThreads == kPTile, "one thread per tile position");
  constexpr int kQuarters = D / 32;
  constexpr int kRotShift = D == 128 ? 1 : 2;  // log2(positions per 128 code bytes)
  {
    const int n = tid;
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
  // V^: item (4 channels c..c+3, 8 positions = 4 token-pair rows): a 4-byte
  // code load per pair row (each byte pairs the row's two positions), the
  // pair's scales, one 16-byte store per channel
#pragma unroll 2
  for (int it = tid; it < (D / 4) * (kPTile / 8); it += kPThreads) {
    const int c = (it % (D / 4)) * 4;
    const int kb = it / (D / 4);
    const int n0 = kb * 8;
    const uint32_t grp = stage + (uint32_t)((n0 / GT) * kGroupBytes);
    uint32_t words[4], sc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + 2 * q;  // even position of the pair
      const int i = (n % GT) >> 1;
      words[q] = 0u;
      sc[q] = 0u;
      if (n < valid) {
        const int phys = (D == 64) ? 8 * ((c >> 3) ^ (((i >> 1) & 1) << 2)) + (c & 7)
                                   : 16 * ((c >> 4) ^ ((i & 3) << 1)) + (c & 15);
        words[q] = lds32(grp + (uint32_t)(GT * (D / 2 + NB) + i * D + phys));
        uint32_t s2 = lds16(grp + (uint32_t)(GT * (D + NB) + i * 2 * NB + 2 * (c >> 4)));
        if (n + 1 >= valid) s2 &= 0x00FFu;  // the pair's second position is past the end: scale 0
        sc[q] = f16x2_from_e4m3x2(s2);
      }
    }
    // the 8 lanes of a store phase write channels 4t + cc: rotating each
    // thread's byte order by (c / 8) mod 4 spreads them over 8 bank groups
    const uint32_t rot = (uint32_t)(c >> 3) & 3u;
    const uint32_t sel = (0x3210u + rot * 0x1111u) & 0x3333u;
    uint32_t r[4][4];  // [rotated channel][pair]
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t t[4];
      f16x2x4_from_e2m1x8(prmt(words[q], 0u, sel), t);  // t[cc]: channel c + (cc + rot) % 4, positions (n, n+1)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) r[cc][q] = hmul2_u32(t[cc], sc[q]);
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      sts128(vdst + core_offset((uint32_t)c + ((cc + rot) & 3u), (uint32_t)n0, D),
             make_uint4(r[cc][0], r[cc][1], r[cc][2], r[cc][3]));
  }
}

template <int D, int GT>
__global__ void __launch_bounds__(kPThreads, 1) prefill_fp4_kernel(const PrefillParams p) {
  using G = PGeo<D>;
  extern __shared__ uint8_t psm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(psm_raw) + 127) & ~uintptr_t(127));
  const uint32_t sb = smem_addr(base);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + G::kBars);
  const uint32_t full0 = smem_addr(full), mma_bar = smem_addr(full + 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 3);
  int* abort = reinterpret_cast<int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int qpb = kPRows / p.g;  // query tokens per CTA
  const int nqb = (p.chunk + qpb - 1) / qpb;
  const int qb = (int)(blockIdx.x % nqb);
  const int bh = (int)(blockIdx.x / nqb);
  const int h = bh % p.hkv, b = bh / p.hkv;
  const int32_t T = __ldg(p.lens + b);
  // this thread's row: query token ti of the chunk, query head hh
  const int ti = qb * qpb + tid / p.g;
  const int hh = h * p.g + tid % p.g;
  const bool row_ok = ti < p.chunk;
  float* orow = p.out + (((int64_t)b * p.chunk + ti) * p.hq + hh) * D;
  if (T < p.chunk) {  // the chunk's own tokens must be in the cache
    if (tid == 0) set_flag(p.flag, KVQ_FLAG_BAD_LENGTH);
    if (row_ok)
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t pos_r = (int64_t)T - p.chunk + ti;  // last position this row attends
  const int last_ti = min(p.chunk, (qb + 1) * qpb) - 1;
  const int ntiles = (int)(((int64_t)T - p.chunk + last_ti) / kPTile) + 1;

  if (tid == 0) {
    mbar_init(full0, 1);
    mbar_init(full0 + 8, 1);
    mbar_init(mma_bar, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);

  // query row -> f16 with a power-of-two prescale (exact for bf16 values in
  // range), into the A-operand layout; the factor returns in the score scale
  float cs = 0.0f;
  {
    float v[D];
    float amax = 0.0f;
    if (row_ok) {
      const uint16_t* src = p.q + (((int64_t)b * p.chunk + ti) * p.hq + hh) * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
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
      for (int i = 0; i < D; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < D; ++i) amax = fmaxf(amax, fabsf(v[i]));
    int k = 0;
    if (amax > 0.0f && amax <= 3.4e38f) {
      const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
      k = min(100, max(-113, 14 - e));
    }
    const float up = __uint_as_float((uint32_t)(k + 127) << 23);
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
      uint32_t f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = pack_f16x2(v[8 * c8 + 2 * j] * up, v[8 * c8 + 2 * j + 1] * up);
      sts128(sb + G::kQ + core_offset((uint32_t)tid, (uint32_t)(c8 * 8), kPRows), make_uint4(f[0], f[1], f[2], f[3]));
    }
    const float sk = p.k_gscale ? __ldg(p.k_gscale + h) : 1.0f;
    cs = p.qk_log2 * sk * __uint_as_float((uint32_t)(127 - k) << 23);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
  const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lanes

  if (tid == 0) {
    issue_tile<D, GT>(p, b, h, 0, T, sb + G::kStage, full0);
    if (ntiles > 1) issue_tile<D, GT>(p, b, h, 1, T, sb + G::kStage + G::kTileBytes, full0 + 8);
  }

  float m_run = -INFINITY, l_run = 0.0f;
  uint32_t mma_phase = 0;
  bool ok = true;
  for (int j = 0; j < ntiles && ok; ++j) {
    const int s = j & 1;
    const uint32_t stage = sb + G::kStage + s * G::kTileBytes;
    ok = mbar_wait(full0 + 8 * s, (j >> 1) & 1);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    dequant_tile<D, GT>(stage, sb + G::kK, sb + G::kV, min((int64_t)kPTile, (int64_t)T - (int64_t)j * kPTile));
    fence_async_smem();
    tc_fence_before();
    __syncthreads();  // K^/V^ written; stage s consumed
    tc_fence_after();
    if (tid == 0) {
      if (j + 2 < ntiles) issue_tile<D, GT>(p, b, h, j + 2, T, stage, full0 + 8 * s);
      constexpr uint32_t kS = idesc_f16_f32(kPRows, kPTile);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc_mma_f16(tmem, smem_desc(sb + G::kQ + ks * 2 * (kPRows / 8) * 128, (kPRows / 8) * 128, 128),
                   smem_desc(sb + G::kK + ks * 2 * (kPTile / 8) * 128, (kPTile / 8) * 128, 128), kS, ks > 0);
      tc_commit(mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(mma_bar, mma_phase & 1));
    ++mma_phase;
    tc_fence_after();
    if (!ok) break;

    // ---- softmax of row tid over this tile, in one pass against the running
    // reference m_run; a row whose tile maximum passes it by the slack (and
    // every row on its first tile) redoes the pass with the raised reference
    const int64_t p0 = (int64_t)j * kPTile;
    const bool all_in = row_ok && p0 + kPTile - 1 <= pos_r;  // no position of the tile masked
    const bool none_in = !row_ok || p0 > pos_r;
    float mt = -INFINITY, lt = 0.0f;
    {
      const float nref = m_run == -INFINITY ? 0.0f : -m_run;
#pragma unroll
      for (int c0 = 0; c0 < kPTile; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_row + (uint32_t)c0, v);
        uint32_t f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float xa = __uint_as_float(v[2 * i]) * cs, xb = __uint_as_float(v[2 * i + 1]) * cs;
          if (!all_in) {
            if (none_in || p0 + c0 + 2 * i > pos_r) xa = -INFINITY;
            if (none_in || p0 + c0 + 2 * i + 1 > pos_r) xb = -INFINITY;
          }
          mt = fmaxf(mt, fmaxf(xa, xb));
          const float pa = fast_exp2(xa + nref), pb = fast_exp2(xb + nref);
          lt += pa + pb;
          f[i] = pack_f16x2(pa, pb);
        }
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
          sts128(sb + G::kP + core_offset((uint32_t)tid, (uint32_t)(c0 + 8 * c8), kPRows),
                 make_uint4(f[4 * c8], f[4 * c8 + 1], f[4 * c8 + 2], f[4 * c8 + 3]));
      }
    }
    const bool raise = row_ok && mt > m_run + kPSlack;
    if (__any_sync(0xFFFFFFFFu, raise)) {
      const float nref = -mt;
#pragma unroll
      for (int c0 = 0; c0 < kPTile; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_row + (uint32_t)c0, v);
        if (raise) {
          uint32_t f[16];
          float l2 = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float xa = __uint_as_float(v[2 * i]) * cs, xb = __uint_as_float(v[2 * i + 1]) * cs;
            if (!all_in) {
              if (p0 + c0 + 2 * i > pos_r) xa = -INFINITY;
              if (p0 + c0 + 2 * i + 1 > pos_r) xb = -INFINITY;
            }
            const float pa = fast_exp2(xa + nref), pb = fast_exp2(xb + nref);
            l2 += pa + pb;
            f[i] = pack_f16x2(pa, pb);
          }
          lt = c0 == 0 ? l2 : lt + l2;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8)
            sts128(sb + G::kP + core_offset((uint32_t)tid, (uint32_t)(c0 + 8 * c8), kPRows),
                   make_uint4(f[4 * c8], f[4 * c8 + 1], f[4 * c8 + 2], f[4 * c8 + 3]));
        }
      }
    }
    // rows that raised their reference: rescale l and their row of O (TMEM
    // accesses are warp-collective; the other rows multiply by 1)
    const float al = (raise && m_run != -INFINITY) ? fast_exp2(m_run - mt) : 1.0f;
    if (__any_sync(0xFFFFFFFFu, al != 1.0f)) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_row + (uint32_t)(kPTile + c0), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
        tmem_st32(t_row + (uint32_t)(kPTile + c0), o);
      }
    }
    if (raise) {
      l_run *= al;
      m_run = mt;
    }
    l_run += lt;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();  // P written; O rescales done
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t kO = idesc_f16_f32(kPRows, D);
#pragma unroll
      for (int ks = 0; ks < kPTile / 16; ++ks)
        tc_mma_f16(tmem + kPTile, smem_desc(sb + G::kP + ks * 2 * (kPRows / 8) * 128, (kPRows / 8) * 128, 128),
                   smem_desc(sb + G::kV + ks * 2 * (D / 8) * 128, (D / 8) * 128, 128), kO, j > 0 || ks > 0);
      tc_commit(mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(mma_bar, mma_phase & 1));
    ++mma_phase;
    tc_fence_after();
  }
  if (ok) {
    const float vs = p.v_gscale ? __ldg(p.v_gscale + h) : 1.0f;
    const float inv = l_run > 0.0f ? vs / l_run : 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      tmem_ld32(t_row + (uint32_t)(kPTile + c0), o);
      if (row_ok) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(orow + c0 + i) =
              make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                          __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
      }
    }
  } else {
    if (tid == 0) {
      set_flag(p.flag, KVQ_FLAG_TIMEOUT);
      // let copies still in flight land before the CTA's shared memory goes away
      for (int s = 0; s < 2; ++s) (void)mbar_try_wait_hint(full0 + 8 * s, 0u, 1000000u);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
  if (g > 8 || (kPRows % g) != 0) return KVQ_ERR_UNSUPPORTED;
  const int64_t nqb = ((int64_t)chunk + kPRows / g - 1) / (kPRows / g);
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
